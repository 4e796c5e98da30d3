"""KV-cache sizing arithmetic -- TEST INFRASTRUCTURE ONLY (part of the oracle).

* Bytes per token = 2 (K and V) x layers L x KV heads H_kv x head dim d x element
  bytes b ["Basics of LLM Inference and vLLM Internals", s.2 "KV Cache and Sizing
  Formulas"; drpranayjha.com, sizing snippet under "How PagedAttention pages the
  KV cache"].
* A request of n tokens occupies ceil(n / block_size) blocks and only its last
  block may be partly filled ["Basics of LLM Inference ...", s.4; "The Memory
  Trick Behind Fast LLM Serving", "PagedAttention changes the shape of the
  problem"].
"""


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def num_logical_blocks(num_tokens: int, block_size: int = 16) -> int:
    return -(-num_tokens // block_size)


def last_block_fill(num_tokens: int, block_size: int = 16) -> int:
    """Tokens held by the last block (0 for an empty request)."""
    if num_tokens == 0:
        return 0
    return num_tokens - (num_logical_blocks(num_tokens, block_size) - 1) * block_size
