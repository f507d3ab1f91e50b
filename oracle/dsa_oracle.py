"""Plain float64 CPU oracle of the DSA decode path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.  It shares
no code with the CUDA library.

What it computes, and where the pages define it:

* ``indexer_logits`` -- the lightning-indexer score
  I[t, s] = sum_j w[t, j] * ReLU(q^I[t, j] . k^I[s])  over 64 FP8 heads of
  128 dims ("MTP and sparse attention: NSA and DSA", section "Sparse
  attention: NSA and DSA").  The FP8 values are dequantised with their
  per-token fp32 scales (the same page: "the indexer key (FP8 + scale)").
* ``visible_lengths`` -- with n_q query tokens per request over S cached
  tokens, query i sees S - (n_q - 1 - i) tokens ("[SGLang] NSA (Narrow Sparse
  Attention)", section "init_forward_metadata": seqlens_expanded, worked
  example 3 queries over 10 tokens -> 8, 9, 10).
* ``topk`` -- per query token, the k = 2048 highest-scoring visible tokens
  ("Sparse attention: NSA and DSA"; "Multi-layer Indexer" abstract).  Ties go
  to the lower token index; the result is a set, returned sorted.
* ``sparse_mla`` -- absorbed-form MLA attention over only the selected latent
  rows: K is the 576-dim latent row, V its first 512 dims ("[SGLang] NSA",
  section "forward_decode": q_nope 512 + q_rope 64, kv_cache_dim =
  kv_lora_rank + qk_rope_head_dim).
* ``sparse_mla_split`` / ``merge`` -- the selected tokens cut into blocks; per
  block an online softmax giving Mid_O and Mid_O_LogExpSum; then a cross-block
  online-softmax merge ("Deepseek Details", section "DSA", stages 2 and 3).
* ``decode_bytes`` / ``decode_flops`` -- the per-layer cost model printed in
  "Sparse attention: NSA and DSA" (its code cell and output table).
* ``encode_e4m3`` / ``quantize_index_key`` / ``cache_write`` -- the step before
  the indexer: each new token's latent row is written into the paged MLA
  cache at its position ("[SGLang] NSA", section "forward_decode":
  set_mla_kv_buffer before the attention), and its indexer key is stored as
  FP8 with one fp32 scale per token ("Sparse attention: NSA and DSA": the
  indexer key, FP8 + scale; "[SGLang] NSA", module list: quant_k_cache, the
  NSA-specific FP8 quantisation of the K cache).  The pages do not give the
  scale rule; the reading here is scale = amax / 448 over the token's 128
  values (448 being E4M3's largest finite magnitude), in fp32.
* ``quantize_latent`` / ``dequantize_latent`` / ``sparse_mla_fp8`` -- the
  latent cache kept in FP8 for the attention ("[SGLang] NSA", its module
  list: quant_k_cache / dequant_k_cache, NSA's own FP8 quantisation of the
  cache, which the attention reads as FP8 to save memory bandwidth).  The
  pages give the format only as E4M3 with fine-grained scaling in 1 x 128
  tiles ("Deepseek Details", section "FP8 Training": activations scaled per
  1 x 128 tile, E4M3 throughout).  Reading: each row's 512 value
  dims are four 128-dim tiles, each E4M3 with one fp32 scale (amax / 448, the
  index key's rule); the 64 rope dims stay bf16 (576 is not a multiple of
  128, and they are no value dims).  A row is 656 bytes: 512 codes, the four
  scales, the 64 rope values.  The attention over such rows is the attention
  over their dequantised values code x scale.

Pinned by ``tests/test_oracle_pins.py``: every function above is checked
against something other than itself (the pages' printed numbers and worked
example, torch's FP8/bf16 conversions, torch's float64 scaled-dot-product
attention, brute-force sorting, invariances and closed forms).
"""
from __future__ import annotations

import math

import numpy as np

PAGE_SIZE = 64
INDEX_HEADS = 64
INDEX_DIM = 128
LATENT_DIM = 576
V_DIM = 512
LATENT_FP8_BYTES = 656   # 512 E4M3 codes + 4 fp32 scales + 64 bf16 rope values

__all__ = [
    "PAGE_SIZE", "INDEX_HEADS", "INDEX_DIM", "LATENT_DIM", "V_DIM",
    "LATENT_FP8_BYTES", "quantize_latent", "dequantize_latent", "sparse_mla_fp8", "attend_fp8",
    "e4m3_table", "decode_e4m3", "decode_bf16", "encode_e4m3", "quantize_index_key",
    "new_token_positions", "cache_write", "visible_lengths",
    "physical_rows", "indexer_logits", "indexer_logits_at", "topk", "attend",
    "selection_count", "split_bounds", "sparse_mla", "sparse_mla_split",
    "merge", "decode_layer", "pair_flops_mla", "pair_flops_indexer",
    "token_bytes_latent", "token_bytes_index", "decode_bytes",
    "decode_flops", "dense_decode_bytes", "dense_decode_flops",
    "layer_bytes", "layer_flops",
]


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def _e4m3_value(b: int) -> float:
    """OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is
    no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    sign = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3 = np.array([_e4m3_value(b) for b in range(256)], dtype=np.float64)


def e4m3_table() -> np.ndarray:
    return _E4M3.copy()


def decode_e4m3(u8: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bytes -> float64 (exact)."""
    return _E4M3[np.asarray(u8, dtype=np.uint8)]


def decode_bf16(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of fp32)."""
    bits = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """Real values -> E4M3 bytes: the nearest finite E4M3 value, ties to the
    code with an even mantissa, magnitudes beyond 448 saturated to 448, the
    sign kept (also for zero).  NaN inputs are not defined here."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    codes = np.arange(0x7F, dtype=np.int64)            # 0x00..0x7E: the finite magnitudes, ascending
    vals = _E4M3[codes]
    hi = np.clip(np.searchsorted(vals, mag, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = np.abs(mag - vals[lo]), np.abs(vals[hi] - mag)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo])
    out = np.where(mag >= 448.0, 0x7E, out)             # saturate
    return (out | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def quantize_index_key(k_bits: np.ndarray):
    """One token's indexer key, [..., 128] bf16 bit patterns -> (E4M3 codes,
    fp32 scale per token).  In fp32: amax = max |k|; scale = amax / 448;
    codes = E4M3(k / scale).  A token of zeros gets scale 1 and zero codes."""
    k = (np.asarray(k_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.max(np.abs(k), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    x = (k / scale[..., None]).astype(np.float32)
    return encode_e4m3(x), scale


def quantize_latent(kv_bits: np.ndarray) -> np.ndarray:
    """Latent rows, [n, 576] bf16 bit patterns -> [n, 656] bytes: the 512
    value dims as four 128-dim tiles of E4M3 codes (each tile quantised like
    an index key: scale = amax / 448 in fp32), then the four fp32 scales
    (little-endian), then the 64 rope dims' bf16 bit patterns (little-endian)."""
    kv = np.asarray(kv_bits, dtype=np.uint16).reshape(-1, LATENT_DIM)
    n = kv.shape[0]
    codes, scales = quantize_index_key(kv[:, :V_DIM].reshape(n, 4, 128))
    out = np.empty((n, LATENT_FP8_BYTES), dtype=np.uint8)
    out[:, :V_DIM] = codes.reshape(n, V_DIM)
    out[:, V_DIM:V_DIM + 16] = scales.astype("<f4").reshape(n, 4).view(np.uint8)
    out[:, V_DIM + 16:] = np.ascontiguousarray(kv[:, V_DIM:]).astype("<u2").view(np.uint8)
    return out


def dequantize_latent(kv8: np.ndarray) -> np.ndarray:
    """[n, 656] FP8 latent rows -> float64 [n, 576]: code x its tile's scale
    for the value dims, the rope dims as they are."""
    kv8 = np.asarray(kv8, dtype=np.uint8).reshape(-1, LATENT_FP8_BYTES)
    n = kv8.shape[0]
    scales = np.ascontiguousarray(kv8[:, V_DIM:V_DIM + 16]).view("<f4").astype(np.float64)
    vals = decode_e4m3(kv8[:, :V_DIM]).reshape(n, 4, 128) * scales[:, :, None]
    rope = decode_bf16(np.ascontiguousarray(kv8[:, V_DIM + 16:]).view("<u2"))
    return np.concatenate([vals.reshape(n, V_DIM), rope], axis=1)


# ---------------------------------------------------------------------------
# Batch geometry
# ---------------------------------------------------------------------------

def visible_lengths(seqlens, q_per_req: int) -> np.ndarray:
    """Tokens visible to each query row, rows ordered request-major.

    Request r holds S_r cached tokens, its q_per_req new tokens included;
    query i of r sees S_r - (q_per_req - 1 - i) of them.
    """
    s = np.asarray(seqlens, dtype=np.int64)
    i = np.arange(q_per_req, dtype=np.int64)
    return (s[:, None] - (q_per_req - 1 - i)[None, :]).reshape(-1)


def physical_rows(page_table_row, positions, page_size: int = PAGE_SIZE) -> np.ndarray:
    """Logical token positions of one request -> rows of the paged cache."""
    pos = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(page_table_row, dtype=np.int64)[pos // page_size]
    return pages * page_size + pos % page_size


def new_token_positions(seqlens, q_per_req: int) -> np.ndarray:
    """Logical position of every new token, rows request-major: request r's
    S_r cached tokens include its q_per_req new ones, which are the last."""
    s = np.asarray(seqlens, dtype=np.int64)
    i = np.arange(q_per_req, dtype=np.int64)
    return (s[:, None] - q_per_req + i[None, :]).reshape(-1)


def cache_write(new_latent, new_index_k, kv, k_fp8, k_scale, page_table, seqlens,
                q_per_req: int):
    """The cache-write step: copies of the caches with every new token's
    latent row written at its position and its indexer key quantised there.

    new_latent [T, 576] and new_index_k [T, 128] are bf16 bit patterns; kv
    [rows, 576] uint16, k_fp8 [rows, 128] uint8, k_scale [rows] float32."""
    kv, k_fp8, k_scale = np.array(kv), np.array(k_fp8), np.array(k_scale)
    pos = new_token_positions(seqlens, q_per_req)
    codes, scales = quantize_index_key(new_index_k)
    for t, p in enumerate(pos):
        r = t // q_per_req
        row = int(physical_rows(page_table[r], [p])[0])
        kv[row] = np.asarray(new_latent[t], dtype=np.uint16)
        k_fp8[row] = codes[t]
        k_scale[row] = scales[t]
    return kv, k_fp8, k_scale


# ---------------------------------------------------------------------------
# Stage 1: lightning indexer
# ---------------------------------------------------------------------------

def indexer_logits_at(q_fp8_t, q_scale_t, w_t, k_fp8, k_scale, rows, with_bound=True):
    """Index scores of one query token against the cache rows ``rows``.

    Returns (I, E): I[s] = sum_j w_j * max(0, qhat_j . khat_s) with
    qhat = e4m3(q) * q_scale and khat = e4m3(k) * k_scale; E[s] is the sum of
    the absolute values of every product in that expression,
    sum_j |w_j| * sum_d |qhat_jd * khat_sd|, the scale of the rounding error.
    """
    qhat = decode_e4m3(q_fp8_t).reshape(INDEX_HEADS, INDEX_DIM) * float(q_scale_t)
    khat = decode_e4m3(k_fp8[rows]).reshape(len(rows), INDEX_DIM) * \
        np.asarray(k_scale, dtype=np.float64)[rows][:, None]
    w = np.asarray(w_t, dtype=np.float64).reshape(INDEX_HEADS)
    dots = khat @ qhat.T                       # [n, 64]
    score = np.maximum(dots, 0.0) @ w          # [n]
    if not with_bound:
        return score, None
    bound = (np.abs(khat) @ np.abs(qhat).T) @ np.abs(w)
    return score, bound


def indexer_logits(q_fp8, q_scale, w, k_fp8, k_scale, page_table, seqlens,
                   q_per_req: int, with_bound: bool = True):
    """Index scores of every query row against its visible tokens.

    Returns (I, E) of shape [T, max_vis]; entries at positions >= the row's
    visible length are -inf in I and 0 in E.
    """
    vis = visible_lengths(seqlens, q_per_req)
    T = vis.shape[0]
    width = int(max(1, vis.max()))
    I = np.full((T, width), -np.inf)
    E = np.zeros((T, width)) if with_bound else None
    for t in range(T):
        r = t // q_per_req
        n = int(vis[t])
        if n <= 0:
            continue
        rows = physical_rows(page_table[r], np.arange(n))
        s, e = indexer_logits_at(q_fp8[t], q_scale[t], w[t], k_fp8, k_scale, rows, with_bound)
        I[t, :n] = s
        if with_bound:
            E[t, :n] = e
    return I, E


# ---------------------------------------------------------------------------
# Stage 2: top-k
# ---------------------------------------------------------------------------

def selection_count(vis, k: int) -> np.ndarray:
    """How many tokens a query selects: all of them when it sees <= k."""
    return np.minimum(np.maximum(np.asarray(vis, dtype=np.int64), 0), k)


def topk(scores, vis, k: int) -> np.ndarray:
    """Per row, the min(k, vis) visible positions with the largest score.

    ``scores`` are compared exactly as given (pass the fp32 tensor to compare
    with a fp32 kernel); -0.0 and +0.0 are equal; equal scores are ordered by
    lower position first.  Each row of the result lists the selected set in
    ascending position order, padded with -1 to k entries.
    """
    scores = np.asarray(scores)
    vis = np.asarray(vis, dtype=np.int64)
    T = scores.shape[0]
    out = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        n = int(max(vis[t], 0))
        m = min(k, n)
        if m == 0:
            continue
        row = scores[t, :n].astype(np.float64) + 0.0   # -0.0 + 0.0 == +0.0
        pos = np.arange(n)
        order = np.lexsort((pos, -row))                # score desc, then position asc
        out[t, :m] = np.sort(order[:m])
    return out


# ---------------------------------------------------------------------------
# Stage 3: sparse MLA over the selected latent rows
# ---------------------------------------------------------------------------

def _attend(qh, rows_lat, sm_scale):
    """Softmax attention of H query heads over n latent rows.

    qh [H, 576], rows_lat [n, 576] (float64).  K = the 576-dim row, V = its
    first 512 dims.  Returns (O [H, 512], lse [H]) with the natural-log
    log-sum-exp of the scaled logits; n == 0 gives O = 0, lse = -inf.
    """
    H = qh.shape[0]
    if rows_lat.shape[0] == 0:
        return np.zeros((H, V_DIM)), np.full(H, -np.inf)
    x = sm_scale * (qh @ rows_lat.T)            # [H, n]
    m = x.max(axis=1, keepdims=True)
    p = np.exp(x - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ rows_lat[:, :V_DIM]) / l
    return o, (m + np.log(l))[:, 0]


def attend(q_bits_t, lat_bits, sm_scale):
    """Attention of one query row (bf16 bits [H, 576]) over the given latent
    rows (bf16 bits [n, 576]): the per-query step of ``sparse_mla``."""
    return _attend(decode_bf16(q_bits_t), decode_bf16(lat_bits).reshape(-1, LATENT_DIM), sm_scale)


def attend_fp8(q_bits_t, kv8_rows, sm_scale):
    """``attend`` over FP8 latent rows ([n, 656] bytes, see quantize_latent)."""
    return _attend(decode_bf16(q_bits_t), dequantize_latent(kv8_rows), sm_scale)


def _selected_rows(idx_row, n_pos, vis_t, page_table_row):
    """Rows of the cache attended by one query: entries at positions < n_pos
    that name a visible token (0 <= idx < vis); other entries are skipped."""
    ids = np.asarray(idx_row[:n_pos], dtype=np.int64)
    ids = ids[(ids >= 0) & (ids < vis_t)]
    return physical_rows(page_table_row, ids)


def _latent_rows(kv_bits, kv_fp8, rows):
    """float64 latent rows of the bf16 cache, or of the FP8 cache if given."""
    if kv_fp8 is not None:
        return dequantize_latent(kv_fp8[rows])
    return decode_bf16(kv_bits[rows])


def sparse_mla(q_bits, kv_bits, idx, page_table, seqlens, q_per_req: int, sm_scale: float,
               tokens=None, kv_fp8=None):
    """Attention of each query row over the tokens its index row selects.

    q_bits [T, H, 576] and kv_bits [rows, 576] are bf16 bit patterns.  Query
    row t reads positions [0, min(k, vis_t)) of idx[t]; entries there that are
    negative or >= vis_t are skipped.  Returns (O [T, H, 512], lse [T, H]).
    ``tokens`` restricts the computation to a subset of rows (others are NaN).
    With ``kv_fp8`` ([rows, 656], see quantize_latent) the rows are read from
    the FP8 cache instead (kv_bits is then unused).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    H = q_bits.shape[1]
    vis = visible_lengths(seqlens, q_per_req)
    n_sel = selection_count(vis, k)
    O = np.full((T, H, V_DIM), np.nan)
    L = np.full((T, H), np.nan)
    for t in (range(T) if tokens is None else tokens):
        r = t // q_per_req
        rows = _selected_rows(idx[t], int(n_sel[t]), int(vis[t]), page_table[r])
        qh = decode_bf16(q_bits[t])
        lat = _latent_rows(kv_bits, kv_fp8, rows)
        O[t], L[t] = _attend(qh, lat, sm_scale)
    return O, L


def sparse_mla_fp8(q_bits, kv_fp8, idx, page_table, seqlens, q_per_req: int, sm_scale: float,
                   tokens=None):
    """sparse_mla over the FP8 latent cache kv_fp8 [rows, 656]."""
    return sparse_mla(q_bits, None, idx, page_table, seqlens, q_per_req, sm_scale, tokens,
                      kv_fp8=kv_fp8)


def split_bounds(k: int, num_splits: int, n_pos: int):
    """Positions [lo, hi) of each split of one query's index row.

    The row's first k positions are cut into num_splits chunks of C
    positions, C = 64 * ceil(ceil(k / num_splits) / 64) (whole 64-token tiles);
    chunk s covers [s*C, (s+1)*C) clipped to the n_pos positions the query
    reads.  (The pages leave the block size open; this is the library's.)
    """
    per = -(-k // num_splits)
    C = 64 * (-(-per // 64))
    out = []
    for s in range(num_splits):
        lo = min(s * C, n_pos)
        hi = min((s + 1) * C, n_pos)
        out.append((lo, hi))
    return out


def sparse_mla_split(q_bits, kv_bits, idx, page_table, seqlens, q_per_req: int,
                     sm_scale: float, num_splits: int, tokens=None, kv_fp8=None):
    """Per-split partial attention: Mid_O [T, H, S, 512] (each block's output
    normalised by its own softmax sum) and Mid_O_LogExpSum [T, H, S].  With
    ``kv_fp8`` the rows come from the FP8 cache."""
    idx = np.asarray(idx)
    T, k = idx.shape
    H = q_bits.shape[1]
    vis = visible_lengths(seqlens, q_per_req)
    n_sel = selection_count(vis, k)
    mid_o = np.full((T, H, num_splits, V_DIM), np.nan)
    mid_l = np.full((T, H, num_splits), np.nan)
    for t in (range(T) if tokens is None else tokens):
        r = t // q_per_req
        qh = decode_bf16(q_bits[t])
        for s, (lo, hi) in enumerate(split_bounds(k, num_splits, int(n_sel[t]))):
            ids = np.asarray(idx[t, lo:hi], dtype=np.int64)
            ids = ids[(ids >= 0) & (ids < vis[t])]
            lat = _latent_rows(kv_bits, kv_fp8, physical_rows(page_table[r], ids))
            mid_o[t, :, s], mid_l[t, :, s] = _attend(qh, lat, sm_scale)
    return mid_o, mid_l


def merge(mid_o, mid_lse):
    """Cross-split online-softmax merge.

    With L = max_s lse_s: O = sum_s exp(lse_s - L) * Mid_O_s / sum_s
    exp(lse_s - L) and lse = L + log(sum_s exp(lse_s - L)).  Splits with
    lse = -inf contribute nothing; if every split is empty, O = 0 and
    lse = -inf.
    """
    mid_o = np.asarray(mid_o, dtype=np.float64)
    mid_lse = np.asarray(mid_lse, dtype=np.float64)
    L = mid_lse.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(L)
    Ls = np.where(empty, 0.0, L)
    wgt = np.where(np.isfinite(mid_lse), np.exp(mid_lse - Ls), 0.0)
    tot = wgt.sum(axis=-1, keepdims=True)
    safe = np.where(tot > 0, tot, 1.0)
    O = (wgt[..., None] * np.where(np.isfinite(mid_lse)[..., None], mid_o, 0.0)).sum(axis=-2) / safe
    lse = np.where(tot > 0, Ls + np.log(safe), -np.inf)[..., 0]
    return O, lse


def decode_layer(inputs: dict, score_dtype=np.float32):
    """The whole decode layer: indexer -> top-k -> sparse MLA.

    The index scores are rounded to ``score_dtype`` before the selection, so
    that the selection is taken in the precision of the scores a kernel
    writes (fp32).  Returns dict(scores, bound, idx, out, lse).
    """
    nq = inputs["q_per_req"]
    I, E = indexer_logits(inputs["q_fp8"], inputs["q_scale"], inputs["w"],
                          inputs["k_fp8"], inputs["k_scale"], inputs["page_table"],
                          inputs["seqlens"], nq)
    vis = visible_lengths(inputs["seqlens"], nq)
    sc = I.astype(score_dtype)
    idx = topk(sc, vis, inputs["topk"])
    out, lse = sparse_mla(inputs["q"], inputs["kv"], idx, inputs["page_table"],
                          inputs["seqlens"], nq, inputs["sm_scale"])
    return dict(scores=I, bound=E, idx=idx, out=out, lse=lse)


# ---------------------------------------------------------------------------
# Cost model ("Sparse attention: NSA and DSA": code cell and output table)
# ---------------------------------------------------------------------------

def pair_flops_mla(num_heads: int = 128, dc: int = 512, rope: int = 64) -> int:
    """Absorbed MLA FLOPs per (query, key): QK over 576 dims + PV over 512."""
    return 2 * num_heads * (dc + rope) + 2 * num_heads * dc


def pair_flops_indexer(heads: int = INDEX_HEADS, dim: int = INDEX_DIM) -> int:
    return 2 * heads * dim


def token_bytes_latent(dc: int = 512, rope: int = 64) -> int:
    return (dc + rope) * 2


def token_bytes_index(dim: int = INDEX_DIM) -> int:
    return dim + 4


def dense_decode_flops(L: int, num_heads: int = 128) -> int:
    return L * pair_flops_mla(num_heads)


def decode_flops(L: int, k: int = 2048, num_heads: int = 128) -> int:
    return L * pair_flops_indexer() + min(L, k) * pair_flops_mla(num_heads)


def dense_decode_bytes(L: int) -> int:
    return L * token_bytes_latent()


def decode_bytes(L: int, k: int = 2048) -> int:
    return L * token_bytes_index() + min(L, k) * token_bytes_latent()


def layer_bytes(seqlens, q_per_req: int, k: int) -> int:
    """Algorithmic HBM bytes of one decode layer over a batch.

    Index keys (128 FP8 bytes + a 4-byte scale per cached token) are read once
    per request and serve all its query tokens; each query token gathers its
    selected latent rows (1152 bytes each).
    """
    vis = visible_lengths(seqlens, q_per_req)
    s = np.asarray(seqlens, dtype=np.int64)
    return int(s.sum() * token_bytes_index() + selection_count(vis, k).sum() * token_bytes_latent())


def layer_flops(seqlens, q_per_req: int, k: int, num_heads: int):
    """(indexer FLOPs, attention FLOPs) of one decode layer over a batch."""
    vis = visible_lengths(seqlens, q_per_req)
    idx = int(np.maximum(vis, 0).sum()) * pair_flops_indexer()
    att = int(selection_count(vis, k).sum()) * pair_flops_mla(num_heads)
    return idx, att
