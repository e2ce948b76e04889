"""Paged KV cache: block-table walk, single-token decode attention, KV append.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, and where the pages say so:

* Paged layout.  K and V of every layer live in fixed-size physical blocks of
  ``block_size`` tokens (16 or 32); a per-sequence block table maps logical
  block j of a sequence to a physical block id.  [SC] "PagedAttention & Memory
  Management (vLLM)" (the logical-to-physical diagram); [FN] "Paged KV-Cache
  with Radix Tree Prefix Cache".  The cache tensors are laid out
  ``[num_blocks, H_kv, block_size, D]`` as in the argument list of the decode
  kernel in [UI] "High-Throughput Paged Attention Kernel Integration".
* Decode.  The one new query token of each sequence attends to all of that
  sequence's cached keys and values: out = softmax(scale * q K^T) V.  [SC]
  "Why We Need the Key-Value (KV) Cache" and "4. Internal workings", step 4;
  the softmax form is [UI] "Mathematical Formulation of Block Salience", the
  definition of A_{l,h,i,j} (there with scale 1/sqrt(D_head)).
* GQA.  Query head hq reads KV head hq // G with G = H_q / H_kv (contiguous
  groups).  [SC] "Attention Architectures: MHA vs. MQA vs. GQA"; the same map
  appears in the [UI] decode kernel (query head divided by the group size).
* Append.  The new token's K/V vectors are written into its slot before the
  token attends.  [SC] "4. Internal workings", step 5, and "Why We Need the
  Key-Value (KV) Cache".  FP8 E4M3 with per-head scaling factors: [FN] FAQ
  "How much HBM memory does FP8 KV-cache quantization save?".

Readings taken where the pages are silent (each is also listed in the design
notes): a slot is ``physical_block * block_size + offset`` and a negative slot
means "skip this row"; ``context_lens`` counts the tokens attended, the
appended token included; a sequence with no tokens yields zeros; FP8 codes are
dequantised as ``value(code) * scale`` with the scale of the (sequence, KV
head) for decode and of the (row, KV head) for append; quantisation divides
by the scale in binary32 and rounds once to E4M3.

This oracle does no splitting and no online softmax: it gathers each sequence
into contiguous K/V and applies the definition.
"""

import numpy as np

from .formats import bf16_bits_to_f64, e4m3_to_f64, e4m3_encode, f32_to_bf16_bits, f32_div

BF16 = "bf16"
F32 = "f32"
E4M3 = "e4m3"


def slot_of(block_table_row, pos, block_size):
    """Flat slot of logical token ``pos`` of one sequence: phys * bs + pos % bs."""
    return int(block_table_row[pos // block_size]) * block_size + pos % block_size


def gather_sequence(cache, block_table_row, ctx, h, block_size):
    """Walk the block table: raw K (or V) rows 0..ctx-1 of KV head ``h``.

    Returns the raw cache words (uint16 bf16 bits or uint8 E4M3 codes) as a
    contiguous ``[ctx, D]`` array, token t taken from
    ``cache[table[t // bs], h, t % bs, :]``.
    """
    t = np.arange(ctx)
    blk = np.asarray(block_table_row)[t // block_size].astype(np.int64)
    off = t % block_size
    return cache[blk, h, off, :]


def dequantize(raw, cache_dtype, scale=None):
    """Exact float64 value of raw cache words (times the FP8 scale if any)."""
    if cache_dtype == BF16:
        return bf16_bits_to_f64(raw)
    if cache_dtype == E4M3:
        return e4m3_to_f64(raw) * np.float64(np.float32(scale))
    raise ValueError(cache_dtype)


def attend(q, K, V, scale):
    """softmax(scale * q K^T) V for query rows q [G, D], K/V [ctx, D], float64."""
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]), dtype=np.float64)
    s = scale * (q @ K.T)                                  # [G, ctx]
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ V                                           # [G, D]


def decode_attention(q_bits, k_cache, v_cache, cache_dtype, block_tables,
                     context_lens, scale, k_scale=None, v_scale=None,
                     units=None):
    """Single-token paged decode attention in float64.

    q_bits        uint16 [B, H_q, D]          bf16 query words
    k/v_cache     [NB, H_kv, bs, D]           uint16 (bf16) or uint8 (E4M3)
    block_tables  int [B, MB]                 entries past the used ones unread
    context_lens  int [B]                     tokens attended per sequence
    scale         float                       softmax scale
    k/v_scale     float32 [B, H_kv]           E4M3 only
    units         optional iterable of (b, h_kv) to compute; others stay NaN

    Returns float64 [B, H_q, D].
    """
    q = bf16_bits_to_f64(q_bits)
    B, H_q, D = q.shape
    NB, H_kv, bs, D2 = k_cache.shape
    assert D2 == D and H_q % H_kv == 0
    G = H_q // H_kv
    out = np.full((B, H_q, D), np.nan)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(H_kv)]
    for b, h in units:
        ctx = int(context_lens[b])
        row = block_tables[b]
        ks = None if k_scale is None else k_scale[b, h]
        vs = None if v_scale is None else v_scale[b, h]
        K = dequantize(gather_sequence(k_cache, row, ctx, h, bs), cache_dtype, ks)
        V = dequantize(gather_sequence(v_cache, row, ctx, h, bs), cache_dtype, vs)
        out[b, h * G:(h + 1) * G] = attend(q[b, h * G:(h + 1) * G], K, V, float(scale))
    return out


def multi_query_attention(q_bits, k_cache, v_cache, cache_dtype, block_tables,
                          context_lens, scale, k_scale=None, v_scale=None, units=None):
    """Paged attention of q_len new tokens per sequence, causal among them.

    The q_len new tokens of sequence b are its last q_len positions
    (context_lens[b] counts them, as for decode): query i sits at position
    p = context_lens[b] - q_len + i and attends tokens 0..p of the sequence,
    i.e. every cached token plus the new tokens up to itself.  Used for a
    chunk of a chunked prefill run next to decode steps ([SC] "9. Failure
    modes and limitations", item 3, Chunked Prefill) and for checking the
    tokens proposed by a draft model in one pass ([SC] "7. Practical
    applications", item 3, Speculative Decoding).  A query with p < 0 (a
    context shorter than q_len) attends nothing and yields zeros, as an empty
    context does for decode.

    q_bits        uint16 [B, q_len, H_q, D]
    other arguments as decode_attention; units: optional (b, h_kv) subset
    Returns float64 [B, q_len, H_q, D].
    """
    q = bf16_bits_to_f64(q_bits)
    B, QL, H_q, D = q.shape
    NB, H_kv, bs, D2 = k_cache.shape
    assert D2 == D and H_q % H_kv == 0
    G = H_q // H_kv
    out = np.full((B, QL, H_q, D), np.nan)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(H_kv)]
    for b, h in units:
        ctx = int(context_lens[b])
        row = block_tables[b]
        ks = None if k_scale is None else k_scale[b, h]
        vs = None if v_scale is None else v_scale[b, h]
        K = dequantize(gather_sequence(k_cache, row, ctx, h, bs), cache_dtype, ks)
        V = dequantize(gather_sequence(v_cache, row, ctx, h, bs), cache_dtype, vs)
        for i in range(QL):
            n = max(ctx - QL + i + 1, 0)
            out[b, i, h * G:(h + 1) * G] = attend(q[b, i, h * G:(h + 1) * G], K[:n], V[:n], float(scale))
    return out


def encode_rows(x, src_dtype, cache_dtype, scale_rows=None):
    """Encode new K or V rows [n, H_kv, D] into cache words.

    bf16 -> bf16 copies the bits; f32 -> bf16 rounds to nearest even;
    {bf16, f32} -> E4M3 divides the binary32 value by the row's scale
    (IEEE binary32 division) and rounds once to E4M3, saturating.
    """
    if src_dtype == BF16:
        xf = bf16_bits_to_f64(x).astype(np.float32)        # exact
        if cache_dtype == BF16:
            return np.asarray(x).astype(np.uint16).copy()
    elif src_dtype == F32:
        xf = np.asarray(x, dtype=np.float32)
        if cache_dtype == BF16:
            return f32_to_bf16_bits(xf)
    else:
        raise ValueError(src_dtype)
    if cache_dtype != E4M3:
        raise ValueError(cache_dtype)
    y = f32_div(xf, np.asarray(scale_rows, dtype=np.float32)[:, :, None])
    return e4m3_encode(y)


def append(k_new, v_new, src_dtype, slot_mapping, k_cache, v_cache, cache_dtype,
           k_scale=None, v_scale=None, scale_row_stride=0):
    """KV append: write row i of k_new/v_new into slot ``slot_mapping[i]``.

    k_new/v_new   [N, H_kv, D]    uint16 bf16 words or float32
    slot_mapping  int [N]         phys * bs + offset; negative = skip
    k/v_cache     [NB, H_kv, bs, D] cache words; NOT modified (copies returned)
    k/v_scale     flat float32; row i, head h uses element i*stride + h
                  (stride 0: one scale per KV head)

    Returns (k_cache', v_cache').
    """
    slots = np.asarray(slot_mapping, dtype=np.int64)
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    NB, H_kv, bs, D = kc.shape
    live = np.nonzero(slots >= 0)[0]
    assert len(np.unique(slots[live])) == len(live), "duplicate slots are undefined"
    if live.size == 0:
        return kc, vc
    assert slots[live].max() < NB * bs
    blk = slots[live] // bs
    off = slots[live] % bs
    ks = vs = None
    if cache_dtype == E4M3:
        idx = live[:, None] * int(scale_row_stride) + np.arange(H_kv)[None, :]
        ks = np.asarray(k_scale, dtype=np.float32).ravel()[idx]
        vs = np.asarray(v_scale, dtype=np.float32).ravel()[idx]
    kc[blk, :, off, :] = encode_rows(np.asarray(k_new)[live], src_dtype, cache_dtype, ks)
    vc[blk, :, off, :] = encode_rows(np.asarray(v_new)[live], src_dtype, cache_dtype, vs)
    return kc, vc
