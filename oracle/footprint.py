"""KV-cache footprint and the capacity arithmetic built on it.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* Footprint.  Total KV bytes = 2 * L * n_kv * d_head * S * B * p, the 2 being
  one tensor for keys and one for values.  [FN] "Quantifying the KV-Cache
  Memory Wall" (Memory_KV); [UI] "The Anatomy of the KV-Cache Memory Wall"
  (M_KV, and M_token = 327,680 bytes per token for L=80, n_kv=8, d=128, p=2).
* Capacity.  The serving simulator of [SC] "6. Implementation: KV Cache Memory
  & Serving Simulator" sizes a cluster: weights in binary GB rounded to two
  decimals, usable pool = total VRAM - weights - per-GPU activation overhead,
  streams = floor(pool bytes / (tokens per stream * KV bytes per token)), and
  the gain of paged over contiguous allocation in whole percent.

Reading taken here: the simulator's printed output for its FP8 run keeps the
weights at 16-bit (only the KV cache is FP8), while its listing would also
halve the weights.  The printed numbers are what the page reports, so the
weight precision is a separate argument.
"""

import math


def kv_bytes(n_layers, n_kv_heads, d_head, seq_len, batch, bytes_per_elem):
    """2 * L * n_kv * d_head * S * B * p bytes."""
    return 2 * n_layers * n_kv_heads * d_head * seq_len * batch * bytes_per_elem


def kv_bytes_per_token(n_layers, n_kv_heads, d_head, bytes_per_elem):
    return kv_bytes(n_layers, n_kv_heads, d_head, 1, 1, bytes_per_elem)


def _round_half_up(x):
    """The simulator rounds halves upwards (towards +infinity)."""
    return math.floor(x + 0.5)


def weights_gb(params_billion, weight_bytes):
    """Weights in binary GB, rounded to two decimals."""
    return _round_half_up(params_billion * 1e9 * weight_bytes / 1024 ** 3 * 100) / 100


def cluster_capacity(params_billion, n_layers, n_kv_heads, d_head, kv_bytes_per_elem,
                     weight_bytes, gpu_count, vram_per_gpu_gb, overhead_per_gpu_gb,
                     avg_ctx, max_ctx):
    """Streams that fit a cluster's KV pool, contiguous vs paged allocation."""
    wgb = weights_gb(params_billion, weight_bytes)
    usable_gb = max(0.0, gpu_count * vram_per_gpu_gb - wgb - gpu_count * overhead_per_gpu_gb)
    bpt = kv_bytes_per_token(n_layers, n_kv_heads, d_head, kv_bytes_per_elem)
    pool = usable_gb * 1024 ** 3
    contiguous = math.floor(pool / (max_ctx * bpt))
    paged = math.floor(pool / (avg_ctx * bpt))
    gain = _round_half_up((paged - contiguous) / contiguous * 100) if contiguous > 0 else 0
    return {
        "kv_bytes_per_token": bpt,
        "weights_gb": wgb,
        "usable_kv_gb": _round_half_up(usable_gb * 10) / 10,
        "streams_contiguous": contiguous,
        "streams_paged": paged,
        "gain_percent": gain,
    }
