"""Byte and FLOP closed forms of the sparse-MLA decode path.

From the footnotes of "vLLM Part 2: PCP/DCP and P/D deployment with HiSparse":
each selected row costs the 656-byte FP8 KV row plus a 4-byte index; each head
adds its bf16 query (576 dims) and output (512 dims); QK over 576 dims and PV
over 512 dims cost 2 FLOPs per multiply-add. KV bytes per token of the pages'
model: 78 MLA layers x 656 B, 21 indexer layers x 132 B (128 FP8 values + a
4-byte scale) and 788 B for the MTP layer.
"""

LATENT, ROPE, QK_DIM, V_DIM = 512, 64, 576, 512


def row_bytes(latent=LATENT, group=128, rope=ROPE) -> int:
    """FP8 latent + one fp32 scale per group + bf16 rope."""
    return latent * 1 + (latent // group) * 4 + rope * 2


def bytes_per_selected_row(row=656, index_bytes=4) -> int:
    return row + index_bytes


def flops_per_row_per_head(qk=QK_DIM, v=V_DIM) -> int:
    return 2 * qk + 2 * v


def q_o_bytes_per_head(qk=QK_DIM, v=V_DIM, elem=2) -> int:
    return qk * elem + v * elem


def query_bytes(heads: int, k=2048) -> int:
    return k * bytes_per_selected_row() + heads * q_o_bytes_per_head()


def query_flops(heads: int, k=2048) -> int:
    return heads * k * flops_per_row_per_head()


def flops_per_byte(heads: int, k=2048) -> float:
    return query_flops(heads, k) / query_bytes(heads, k)


def kv_bytes_per_token(mla_layers=78, idx_layers=21, idx_bytes=132, mtp_bytes=788, row=656) -> int:
    return mla_layers * row + idx_layers * idx_bytes + mtp_bytes


def ridge_flops_per_byte(tflops: float, tbps: float) -> float:
    return tflops / tbps
