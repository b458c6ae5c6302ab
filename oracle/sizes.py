"""K/V cache sizes.  TEST INFRASTRUCTURE ONLY (see the package docstring).

[note] 历史背景 ("KV cache 为什么突然成了主角") and [guide] 01 give the size of one
token's K/V cache as 2 (key and value) x hidden size x layers x bytes per
element: for OPT-13B, 2 x 5120 x 40 x 2 bytes, "about 800 KB", and "about
1.6 GB" for a 2048-token request.
"""


def kv_bytes_per_token(num_layers: int, num_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Bytes of K and V one token occupies across all layers (hidden = heads x head_dim)."""
    return 2 * num_layers * num_heads * head_dim * dtype_bytes


def kv_bytes_per_block(num_heads: int, head_dim: int, block_size: int, dtype_bytes: int = 2) -> int:
    """Bytes of one physical block of one layer's K pool (the V pool holds as many)."""
    return num_heads * block_size * head_dim * dtype_bytes
