// dsa_api.cu -- the C ABI of libdsa.so (declared and documented in
// include/dsa.h): argument validation, workspace layout, TMA descriptor
// encoding and the launch sequence of the decode layer.
#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "dsa.h"
#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

namespace {
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_sm_count[64] = {0};
}  // namespace

namespace {
bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_tmap_nd(map, dtype, base, 2, dims, strides, box, swizzle);
}

bool encode_tmap_nd(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                    const uint64_t* dims, const uint64_t* byte_strides, const uint32_t* box,
                    CUtensorMapSwizzle swizzle) {
  if (!load_encoder() || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) st[i] = byte_strides[i];
  }
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int check_decode_desc(const ::dsa_decode_desc* d) {
  if (!d) return ::DSA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->q_per_req < 1 || d->num_heads < 1 || d->topk < 1 || d->max_pages < 1 ||
      d->num_pages < 1)
    return ::DSA_ERR_INVALID_ARG;
  if (!d->seqlens || !d->page_table || (reinterpret_cast<uintptr_t>(d->seqlens) & 3) ||
      (reinterpret_cast<uintptr_t>(d->page_table) & 3))
    return ::DSA_ERR_INVALID_ARG;
  if (d->batch > DSA_MAX_BATCH || d->q_per_req > DSA_MAX_Q_PER_REQ) return ::DSA_ERR_UNSUPPORTED;
  if (d->num_heads > 128 || d->num_heads % 16 != 0) return ::DSA_ERR_UNSUPPORTED;
  if (d->topk > DSA_MAX_TOPK || d->page_size != DSA_PAGE_SIZE) return ::DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->num_pages) * DSA_PAGE_SIZE >= (int64_t(1) << 31) ||
      static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE >= (int64_t(1) << 31))
    return ::DSA_ERR_UNSUPPORTED;
  return ::DSA_OK;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && g_sm_count[dev] > 0) return g_sm_count[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) g_sm_count[dev] = n;
  return n;
}

}  // namespace dsa

namespace {

using dsa::kHistBins;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

dsa_status check_desc(const dsa_decode_desc* d) {
  return static_cast<dsa_status>(dsa::check_decode_desc(d));
}

int rows_of(const dsa_decode_desc* d) { return d->batch * d->q_per_req; }

// Zero-fills n16 16-byte words; lets its dependent (the indexer) start at once.
__global__ void ws_clear_kernel(uint4* p, long long n16) {
  dsa::grid_dep_launch();
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += step)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

int max_splits(const dsa_decode_desc* d) { return (d->topk + 63) / 64; }

int resolve_splits(const dsa_decode_desc* d, int32_t num_splits) {
  return num_splits == 0 ? dsa_num_splits_auto(d) : num_splits;
}

dsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

struct TopkWs {
  size_t hist, cand, total;
};

TopkWs topk_ws_layout(int T, int64_t ld) {
  TopkWs w;
  w.hist = 0;
  w.cand = align256(w.hist + size_t(T) * kHistBins * 4);
  w.total = align256(w.cand + size_t(T) * size_t(ld) * 8);
  return w;
}

struct FusedWs {
  int64_t ld;
  size_t logits, hist, cand, topk, mid_o, mid_lse, total;
};

FusedWs fused_ws_layout(const dsa_decode_desc* d, int32_t max_seqlen, int splits) {
  FusedWs w;
  const int T = rows_of(d);
  w.ld = ((static_cast<int64_t>(max_seqlen) + 127) / 128) * 128;
  w.logits = 0;
  w.hist = align256(w.logits + size_t(T) * size_t(w.ld) * 4);
  w.cand = align256(w.hist + size_t(T) * kHistBins * 4);
  w.topk = align256(w.cand + size_t(T) * size_t(w.ld) * 8);
  w.mid_o = align256(w.topk + size_t(T) * size_t(d->topk) * 4);
  const size_t mo = splits > 1 ? size_t(T) * d->num_heads * splits * dsa::kVDim * 4 : 0;
  w.mid_lse = align256(w.mid_o + mo);
  w.total = align256(w.mid_lse + size_t(T) * d->num_heads * splits * 4);
  return w;
}

}  // namespace

extern "C" {

const char* dsa_status_str(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_version(void) { return "dsa-gb300 0.2 (sm_103a)"; }

dsa_status dsa_debug_set_wait_cycles(int64_t cycles) {
  if (cycles < 0) return DSA_ERR_INVALID_ARG;
  dsa::set_indexer_wait_cycles(cycles);
  return DSA_OK;
}

int32_t dsa_num_splits_auto(const dsa_decode_desc* d) {
  if (!d || d->batch < 1 || d->q_per_req < 1 || d->topk < 1) return 1;
  // As many CTA pairs per query row as fill the SMs, then the fewest splits
  // that keep the same number of 64-key tiles per split (no empty splits).
  const int T = rows_of(d);
  const int sms = dsa::device_sm_count();
  const int tiles = max_splits(d);
  int s = sms / (2 * T);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  const int per = (tiles + s - 1) / s;
  return (tiles + per - 1) / per;
}

dsa_status dsa_indexer_logits(const dsa_decode_desc* d, const uint8_t* q_fp8, const float* q_scale,
                              const float* w, const uint8_t* k_fp8, const float* k_scale,
                              float* logits, int64_t ld, void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!q_fp8 || !q_scale || !w || !k_fp8 || !k_scale || !logits) return DSA_ERR_INVALID_ARG;
  if (!aligned(q_fp8, 16) || !aligned(k_fp8, 16) || !aligned(logits, 16) || !aligned(q_scale, 4) ||
      !aligned(w, 4) || !aligned(k_scale, 16))
    return DSA_ERR_INVALID_ARG;
  if (ld < static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE || ld % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  dsa::IndexerLaunch a{};
  a.q_fp8 = q_fp8; a.q_scale = q_scale; a.w = w; a.k_fp8 = k_fp8; a.k_scale = k_scale;
  a.seqlens = d->seqlens; a.page_table = d->page_table; a.logits = logits; a.ld = ld;
  a.hist = nullptr; a.batch = d->batch; a.nq = d->q_per_req; a.max_pages = d->max_pages;
  a.num_pages = d->num_pages; a.topk = d->topk; a.skip_short = 0;
  return cuda_status(dsa::launch_indexer(a, static_cast<cudaStream_t>(stream)));
}

size_t dsa_topk_workspace_bytes(const dsa_decode_desc* d, int64_t ld) {
  if (!d || d->batch < 1 || d->q_per_req < 1 || ld < 1) return 0;
  return topk_ws_layout(rows_of(d), ld).total;
}

dsa_status dsa_topk(const dsa_decode_desc* d, const float* logits, int64_t ld, int32_t* topk_idx,
                    void* ws, size_t ws_bytes, void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!logits || !topk_idx || !aligned(logits, 16) || !aligned(topk_idx, 4))
    return DSA_ERR_INVALID_ARG;
  if (ld < static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE || ld % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  if (ld > dsa::kTopkMaxLd) return DSA_ERR_UNSUPPORTED;
  const TopkWs lay = topk_ws_layout(rows_of(d), ld);
  if (!ws || !aligned(ws, 16) || ws_bytes < lay.total) return DSA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaError_t e = cudaMemsetAsync(base + lay.hist, 0, lay.cand - lay.hist, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  dsa::TopkLaunch a{};
  a.seqlens = d->seqlens; a.logits = logits; a.ld = ld; a.out = topk_idx;
  a.hist = reinterpret_cast<uint32_t*>(base + lay.hist);
  a.cand = reinterpret_cast<uint2*>(base + lay.cand);
  a.batch = d->batch; a.nq = d->q_per_req; a.k = d->topk; a.hist_ready = 0;
  return cuda_status(dsa::launch_topk(a, s));
}

namespace {

// The attention stage over the bf16 cache kv, or over the FP8 cache kv8.
dsa_status mla_split(const dsa_decode_desc* d, const uint16_t* q, const uint16_t* kv,
                     const uint8_t* kv8, const int32_t* topk_idx, int32_t num_splits,
                     float sm_scale, float* mid_o, float* mid_lse, void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!q || (!kv && !kv8) || !topk_idx || !mid_o || !mid_lse) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || (kv && !aligned(kv, 16)) || (kv8 && !aligned(kv8, 16)) ||
      !aligned(mid_o, 16) || !aligned(topk_idx, 4) || !aligned(mid_lse, 4))
    return DSA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  const int splits = resolve_splits(d, num_splits);
  if (splits < 1 || splits > max_splits(d)) return DSA_ERR_INVALID_ARG;
  dsa::MlaLaunch a{};
  a.q = q; a.kv = kv; a.kv8 = kv8; a.topk_idx = topk_idx; a.seqlens = d->seqlens;
  a.page_table = d->page_table;
  a.mid_o = mid_o; a.mid_lse = mid_lse; a.batch = d->batch; a.nq = d->q_per_req;
  a.heads = d->num_heads; a.k = d->topk; a.max_pages = d->max_pages; a.num_pages = d->num_pages;
  a.num_splits = splits; a.sm_scale = sm_scale;
  return cuda_status(dsa::launch_sparse_mla(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

dsa_status dsa_sparse_mla_decode_split(const dsa_decode_desc* d, const uint16_t* q,
                                       const uint16_t* kv, const int32_t* topk_idx,
                                       int32_t num_splits, float sm_scale, float* mid_o,
                                       float* mid_lse, void* stream) {
  if (!kv) return DSA_ERR_INVALID_ARG;
  return mla_split(d, q, kv, nullptr, topk_idx, num_splits, sm_scale, mid_o, mid_lse, stream);
}

dsa_status dsa_sparse_mla_decode_split_fp8(const dsa_decode_desc* d, const uint16_t* q,
                                           const uint8_t* kv8, const int32_t* topk_idx,
                                           int32_t num_splits, float sm_scale, float* mid_o,
                                           float* mid_lse, void* stream) {
  if (!kv8) return DSA_ERR_INVALID_ARG;
  return mla_split(d, q, nullptr, kv8, topk_idx, num_splits, sm_scale, mid_o, mid_lse, stream);
}

dsa_status dsa_latent_to_fp8(const uint16_t* kv, int64_t rows, uint8_t* kv8, void* stream) {
  if (rows < 0) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!kv || !kv8 || !aligned(kv, 16) || !aligned(kv8, 16)) return DSA_ERR_INVALID_ARG;
  return cuda_status(dsa::launch_latent_fp8(kv, rows, kv8, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_merge(int32_t num_rows, int32_t num_splits, const float* mid_o, const float* mid_lse,
                     float* out, float* out_lse, void* stream) {
  if (num_rows < 0 || num_splits < 1) return DSA_ERR_INVALID_ARG;
  if (num_splits > 32) return DSA_ERR_UNSUPPORTED;
  if (num_rows == 0) return DSA_OK;
  if (!mid_o || !mid_lse || !out || !aligned(mid_o, 16) || !aligned(out, 16) ||
      !aligned(mid_lse, 4) || (out_lse && !aligned(out_lse, 4)))
    return DSA_ERR_INVALID_ARG;
  return cuda_status(dsa::launch_merge(num_rows, num_splits, mid_o, mid_lse, out, out_lse,
                                       static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_cache_write(const dsa_decode_desc* d, const uint16_t* new_latent,
                           const uint16_t* new_index_k, uint16_t* kv, uint8_t* k_fp8, float* k_scale,
                           void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!new_latent || !new_index_k || !kv || !k_fp8 || !k_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned(new_latent, 16) || !aligned(kv, 16) || !aligned(new_index_k, 8) ||
      !aligned(k_fp8, 4) || !aligned(k_scale, 4))
    return DSA_ERR_INVALID_ARG;
  dsa::CacheWriteLaunch a{};
  a.new_latent = new_latent; a.new_index_k = new_index_k; a.kv = kv; a.k_fp8 = k_fp8;
  a.k_scale = k_scale; a.seqlens = d->seqlens; a.page_table = d->page_table;
  a.batch = d->batch; a.nq = d->q_per_req; a.max_pages = d->max_pages; a.num_pages = d->num_pages;
  return cuda_status(dsa::launch_cache_write(a, static_cast<cudaStream_t>(stream)));
}

size_t dsa_workspace_bytes(const dsa_decode_desc* d, int32_t max_seqlen, int32_t num_splits) {
  if (!d || d->batch < 1 || d->q_per_req < 1 || d->topk < 1 || d->num_heads < 1 ||
      max_seqlen < 1 || num_splits < 0)
    return 0;
  return fused_ws_layout(d, max_seqlen, resolve_splits(d, num_splits)).total;
}

dsa_status dsa_decode_fused(const dsa_decode_desc* d, const uint8_t* q_fp8, const float* q_scale,
                            const float* w, const uint8_t* k_fp8, const float* k_scale,
                            const uint16_t* q, const uint16_t* kv, const int32_t* topk_in,
                            int32_t* topk_out, float sm_scale, int32_t num_splits,
                            int32_t max_seqlen, float* out, void* ws, size_t ws_bytes,
                            void* stream) {
  return dsa_decode_fused_timed(d, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, topk_in, topk_out,
                                sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream,
                                nullptr);
}

namespace {

// The layer; with `cw` the new tokens' cache write runs first, in the kernel
// that also clears the workspace (the indexer waits for it only before each
// request's last two tiles).
dsa_status fused_layer(const dsa_decode_desc* d, const dsa::CacheWriteLaunch* cw,
                       const uint8_t* q_fp8, const float* q_scale, const float* w,
                       const uint8_t* k_fp8, const float* k_scale, const uint16_t* q,
                       const uint16_t* kv, const uint8_t* kv8, const int32_t* topk_in,
                       int32_t* topk_out,
                       float sm_scale, int32_t num_splits, int32_t max_seqlen, float* out,
                       void* ws, size_t ws_bytes, void* stream, void* const* stage_events,
                       bool check_only = false) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!q || (!kv && !kv8) || !out || !aligned(q, 16) || (kv && !aligned(kv, 16)) ||
      (kv8 && !aligned(kv8, 16)) || !aligned(out, 16))
    return DSA_ERR_INVALID_ARG;
  if (!topk_in && (!q_fp8 || !q_scale || !w || !k_fp8 || !k_scale || !aligned(q_fp8, 16) ||
                   !aligned(k_fp8, 16) || !aligned(q_scale, 4) || !aligned(w, 4) ||
                   !aligned(k_scale, 16)))
    return DSA_ERR_INVALID_ARG;
  if ((topk_in && !aligned(topk_in, 4)) || (topk_out && !aligned(topk_out, 4)))
    return DSA_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  if (max_seqlen < 1 || static_cast<int64_t>(max_seqlen) > static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE)
    return DSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_seqlen) > dsa::kTopkMaxLd)
    return DSA_ERR_UNSUPPORTED;
  const int splits = resolve_splits(d, num_splits);
  if (splits < 1 || splits > max_splits(d)) return DSA_ERR_INVALID_ARG;
  if (splits > 32) return DSA_ERR_UNSUPPORTED;
  const FusedWs lay = fused_ws_layout(d, max_seqlen, splits);
  if (!ws || !aligned(ws, 256) || ws_bytes < lay.total) return DSA_ERR_WORKSPACE;
  if (check_only) return DSA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int T = rows_of(d);

  auto mark = [&](int i) -> bool {
    return !stage_events || !stage_events[i] ||
           cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s) == cudaSuccess;
  };
  const int32_t* idx = topk_in;
  if (!topk_in) {
    int32_t* sel = topk_out ? topk_out : reinterpret_cast<int32_t*>(base + lay.topk);
    // The histogram starts at zero: a small kernel clears it
    // and the indexer runs as its dependent (prologue and key stream overlap
    // the clear; only its first histogram flush waits for it).
    const long long n16 = static_cast<long long>((lay.cand - lay.hist) / 16);
    cudaError_t e;
    if (cw) {
      dsa::CacheWriteLaunch c = *cw;
      c.clear = reinterpret_cast<uint4*>(base + lay.hist);
      c.clear_n16 = n16;
      e = dsa::launch_cache_write(c, s);
    } else {
      const int cgrid = static_cast<int>(std::min<long long>((n16 + 255) / 256, 148));
      e = dsa::launch_kernel(ws_clear_kernel, dim3(cgrid), dim3(256), 0, s, false, 1,
                             reinterpret_cast<uint4*>(base + lay.hist), n16);
    }
    // Stage 0 (timed entry only) starts after the clear: it times the indexer.
    if (e != cudaSuccess || !mark(0)) return DSA_ERR_CUDA;
    dsa::IndexerLaunch ia{};
    ia.q_fp8 = q_fp8; ia.q_scale = q_scale; ia.w = w; ia.k_fp8 = k_fp8; ia.k_scale = k_scale;
    ia.seqlens = d->seqlens; ia.page_table = d->page_table;
    ia.logits = reinterpret_cast<float*>(base + lay.logits); ia.ld = lay.ld;
    ia.hist = reinterpret_cast<uint32_t*>(base + lay.hist);
    ia.batch = d->batch; ia.nq = d->q_per_req; ia.max_pages = d->max_pages;
    ia.num_pages = d->num_pages; ia.topk = d->topk; ia.skip_short = 1; ia.pdl = 1;
    ia.wait_tail = cw ? 1 : 0;
    e = dsa::launch_indexer(ia, s);
    if (e != cudaSuccess || !mark(1)) return DSA_ERR_CUDA;
    dsa::TopkLaunch ta{};
    ta.seqlens = d->seqlens; ta.logits = ia.logits; ta.ld = lay.ld; ta.out = sel;
    ta.hist = ia.hist;
    ta.cand = reinterpret_cast<uint2*>(base + lay.cand);
    ta.batch = d->batch; ta.nq = d->q_per_req; ta.k = d->topk; ta.hist_ready = 1;
    ta.pdl = 1;   // overlaps its launch with the indexer's last CTAs
    e = dsa::launch_topk(ta, s);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    idx = sel;
  } else {
    // The attention below is a plain launch: it starts after the write.
    if (cw && dsa::launch_cache_write(*cw, s) != cudaSuccess) return DSA_ERR_CUDA;
    if (!mark(0) || !mark(1)) return DSA_ERR_CUDA;
  }
  if (!mark(2)) return DSA_ERR_CUDA;
  dsa::MlaLaunch ma{};
  ma.q = q; ma.kv = kv; ma.kv8 = kv8; ma.topk_idx = idx; ma.seqlens = d->seqlens; ma.page_table = d->page_table;
  ma.mid_o = splits > 1 ? reinterpret_cast<float*>(base + lay.mid_o) : out;
  ma.mid_lse = reinterpret_cast<float*>(base + lay.mid_lse);
  ma.batch = d->batch; ma.nq = d->q_per_req; ma.heads = d->num_heads; ma.k = d->topk;
  ma.max_pages = d->max_pages; ma.num_pages = d->num_pages; ma.num_splits = splits;
  ma.sm_scale = sm_scale;
  // After the fused top-k, the attention CTAs start (and fetch their queries)
  // while the top-k finishes; they wait for it before reading its rows.
  ma.pdl = topk_in ? 0 : 1;
  cudaError_t e = dsa::launch_sparse_mla(ma, s);
  if (e != cudaSuccess || !mark(3)) return DSA_ERR_CUDA;
  if (splits > 1) {
    // A plain launch: launched early, the merge's CTAs would sit on the
    // attention's SMs (they need no shared memory) while it runs, and the
    // layer measured ~1 us slower.
    e = dsa::launch_merge(T * d->num_heads, splits, ma.mid_o, ma.mid_lse, out, nullptr, s, false);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  if (!mark(4)) return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // namespace

dsa_status dsa_decode_fused_timed(const dsa_decode_desc* d, const uint8_t* q_fp8,
                                  const float* q_scale, const float* w, const uint8_t* k_fp8,
                                  const float* k_scale, const uint16_t* q, const uint16_t* kv,
                                  const int32_t* topk_in, int32_t* topk_out, float sm_scale,
                                  int32_t num_splits, int32_t max_seqlen, float* out, void* ws,
                                  size_t ws_bytes, void* stream, void* const* stage_events) {
  return fused_layer(d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, topk_in,
                     topk_out, sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream,
                     stage_events);
}

dsa_status dsa_decode_fused_write(const dsa_decode_desc* d, const uint16_t* new_latent,
                                  const uint16_t* new_index_k, const uint8_t* q_fp8,
                                  const float* q_scale, const float* w, uint8_t* k_fp8,
                                  float* k_scale, const uint16_t* q, uint16_t* kv,
                                  const int32_t* topk_in, int32_t* topk_out, float sm_scale,
                                  int32_t num_splits, int32_t max_seqlen, float* out, void* ws,
                                  size_t ws_bytes, void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!new_latent || !new_index_k || !kv || !k_fp8 || !k_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned(new_latent, 16) || !aligned(new_index_k, 8) || !aligned(k_fp8, 4) ||
      !aligned(k_scale, 4))
    return DSA_ERR_INVALID_ARG;
  dsa::CacheWriteLaunch c{};
  c.new_latent = new_latent; c.new_index_k = new_index_k; c.kv = kv; c.k_fp8 = k_fp8;
  c.k_scale = k_scale; c.seqlens = d->seqlens; c.page_table = d->page_table;
  c.batch = d->batch; c.nq = d->q_per_req; c.max_pages = d->max_pages; c.num_pages = d->num_pages;
  return fused_layer(d, &c, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, topk_in, topk_out,
                     sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream, nullptr);
}

dsa_status dsa_decode_fused_fp8kv(const dsa_decode_desc* d, const uint8_t* q_fp8,
                                  const float* q_scale, const float* w, const uint8_t* k_fp8,
                                  const float* k_scale, const uint16_t* q, const uint8_t* kv8,
                                  const int32_t* topk_in, int32_t* topk_out, float sm_scale,
                                  int32_t num_splits, int32_t max_seqlen, float* out, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!kv8) return DSA_ERR_INVALID_ARG;
  return fused_layer(d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, nullptr, kv8, topk_in,
                     topk_out, sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream, nullptr);
}

int32_t dsa_num_splits_mli(const dsa_decode_desc* d) {
  if (!d || d->batch < 1 || d->q_per_req < 1 || d->topk < 1) return 1;
  // The attention shares the GPU with the top-k, which holds up to ~40 % of
  // the SMs: its CTAs (two per split) take about 58 % of them; then the
  // fewest splits with the same number of 64-key tiles per split.
  const int T = rows_of(d);
  const int sms = dsa::device_sm_count();
  const int tiles = max_splits(d);
  int s = (sms * 7 / 12) / (2 * T);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  const int per = (tiles + s - 1) / s;
  return (tiles + per - 1) / per;
}

dsa_status dsa_decode_mli(const dsa_decode_desc* d, const uint8_t* q_fp8, const float* q_scale,
                          const float* w, const uint8_t* k_fp8, const float* k_scale,
                          const uint16_t* q, const uint16_t* kv, const int32_t* topk_prev,
                          int32_t* topk_next, float sm_scale, int32_t num_splits,
                          int32_t max_seqlen, float* out, void* ws, size_t ws_bytes,
                          void* stream) {
  dsa_status st = check_desc(d);
  if (st != DSA_OK) return st;
  if (!topk_prev || !topk_next || !aligned(topk_prev, 4) || !aligned(topk_next, 4))
    return DSA_ERR_INVALID_ARG;
  const int splits = num_splits == 0 ? dsa_num_splits_mli(d) : num_splits;
  if (splits < 1 || splits > max_splits(d)) return DSA_ERR_INVALID_ARG;
  // The rest as the fused layer checks it (indexer inputs required here).
  st = fused_layer(d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, nullptr, topk_next,
                   sm_scale, splits, max_seqlen, out, ws, ws_bytes, stream, nullptr,
                   /*check_only=*/true);
  if (st != DSA_OK) return st;
  const FusedWs lay = fused_ws_layout(d, max_seqlen, splits);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int T = rows_of(d);

  // 1-3. The layer's own selection, as in the fused layer: the workspace
  //      clear, the indexer (one CTA per SM) as its programmatic dependent,
  //      the top-k as the indexer's, writing topk_next.
  const long long n16 = static_cast<long long>((lay.cand - lay.hist) / 16);
  const int cgrid = static_cast<int>(std::min<long long>((n16 + 255) / 256, 148));
  cudaError_t e = dsa::launch_kernel(ws_clear_kernel, dim3(cgrid), dim3(256), 0, s, false, 1,
                                     reinterpret_cast<uint4*>(base + lay.hist), n16);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  dsa::IndexerLaunch ia{};
  ia.q_fp8 = q_fp8; ia.q_scale = q_scale; ia.w = w; ia.k_fp8 = k_fp8; ia.k_scale = k_scale;
  ia.seqlens = d->seqlens; ia.page_table = d->page_table;
  ia.logits = reinterpret_cast<float*>(base + lay.logits); ia.ld = lay.ld;
  ia.hist = reinterpret_cast<uint32_t*>(base + lay.hist);
  ia.batch = d->batch; ia.nq = d->q_per_req; ia.max_pages = d->max_pages;
  ia.num_pages = d->num_pages; ia.topk = d->topk; ia.skip_short = 1; ia.pdl = 1;
  e = dsa::launch_indexer(ia, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  dsa::TopkLaunch ta{};
  ta.seqlens = d->seqlens; ta.logits = ia.logits; ta.ld = lay.ld; ta.out = topk_next;
  ta.hist = ia.hist;
  ta.cand = reinterpret_cast<uint2*>(base + lay.cand);
  ta.batch = d->batch; ta.nq = d->q_per_req; ta.k = d->topk; ta.hist_ready = 1; ta.pdl = 1;
  e = dsa::launch_topk(ta, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  // 4. The attention over the earlier layer's selection as the top-k's
  //    programmatic dependent: its CTAs start once every top-k CTA runs,
  //    on the SMs the top-k leaves free, and read topk_prev without waiting
  //    (it was complete before this call); its grid completes after the
  //    top-k's.
  dsa::MlaLaunch ma{};
  ma.q = q; ma.kv = kv; ma.kv8 = nullptr; ma.topk_idx = topk_prev; ma.seqlens = d->seqlens;
  ma.page_table = d->page_table;
  ma.mid_o = splits > 1 ? reinterpret_cast<float*>(base + lay.mid_o) : out;
  ma.mid_lse = reinterpret_cast<float*>(base + lay.mid_lse);
  ma.batch = d->batch; ma.nq = d->q_per_req; ma.heads = d->num_heads; ma.k = d->topk;
  ma.max_pages = d->max_pages; ma.num_pages = d->num_pages; ma.num_splits = splits;
  ma.sm_scale = sm_scale; ma.pdl = 1; ma.sel_ready = 1;
  e = dsa::launch_sparse_mla(ma, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  // 5. The merge of the attention's splits.
  if (splits > 1) {
    e = dsa::launch_merge(T * d->num_heads, splits, ma.mid_o, ma.mid_lse, out, nullptr, s, false);
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

namespace {

size_t step_layout(int32_t batch, int32_t q_per_req, int32_t num_heads, int32_t max_pages,
                   dsa_step_layout* L) {
  const size_t T = static_cast<size_t>(batch) * q_per_req;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L->q_fp8 = take(T * DSA_INDEX_HEADS * DSA_INDEX_DIM);
  L->q_scale = take(T * 4);
  L->w = take(T * DSA_INDEX_HEADS * 4);
  L->q = take(T * static_cast<size_t>(num_heads) * DSA_LATENT_DIM * 2);
  L->seqlens = take(static_cast<size_t>(batch) * 4);
  L->page_table = take(static_cast<size_t>(batch) * max_pages * 4);
  L->bytes = off;
  return off;
}

}  // namespace

dsa_status dsa_step_layout_get(int32_t batch, int32_t q_per_req, int32_t num_heads,
                               int32_t max_pages, dsa_step_layout* layout) {
  if (!layout || batch < 1 || q_per_req < 1 || num_heads < 1 || max_pages < 1)
    return DSA_ERR_INVALID_ARG;
  if (batch > DSA_MAX_BATCH || q_per_req > DSA_MAX_Q_PER_REQ || num_heads > 128)
    return DSA_ERR_UNSUPPORTED;
  step_layout(batch, q_per_req, num_heads, max_pages, layout);
  return DSA_OK;
}

dsa_status dsa_decode_step_host(const dsa_decode_desc* desc, const void* host_in, void* dev_in,
                                const uint8_t* k_fp8, const float* k_scale, const uint16_t* kv,
                                float sm_scale, int32_t num_splits, int32_t max_seqlen,
                                float* out, float* host_out, void* ws, size_t ws_bytes,
                                void* stream) {
  if (!desc || !host_in || !dev_in || !aligned(dev_in, 256)) return DSA_ERR_INVALID_ARG;
  dsa_step_layout L;
  dsa_status st = dsa_step_layout_get(desc->batch, desc->q_per_req, desc->num_heads,
                                      desc->max_pages, &L);
  if (st != DSA_OK) return st;
  uint8_t* in = static_cast<uint8_t*>(dev_in);
  dsa_decode_desc d = *desc;
  d.seqlens = reinterpret_cast<const int32_t*>(in + L.seqlens);
  d.page_table = reinterpret_cast<const int32_t*>(in + L.page_table);
  const uint8_t* q_fp8 = in + L.q_fp8;
  const float* q_scale = reinterpret_cast<const float*>(in + L.q_scale);
  const float* w = reinterpret_cast<const float*>(in + L.w);
  const uint16_t* q = reinterpret_cast<const uint16_t*>(in + L.q);
  // Every argument is checked before the first copy is queued.
  st = fused_layer(&d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, nullptr,
                   nullptr, sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream, nullptr,
                   /*check_only=*/true);
  if (st != DSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dev_in, host_in, L.bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  st = fused_layer(&d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, nullptr,
                   nullptr, sm_scale, num_splits, max_seqlen, out, ws, ws_bytes, stream, nullptr);
  if (st != DSA_OK) return st;
  if (host_out) {
    const size_t ob = static_cast<size_t>(rows_of(&d)) * d.num_heads * DSA_V_DIM * sizeof(float);
    if (cudaMemcpyAsync(host_out, out, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

dsa_status dsa_decode_step_ring(const dsa_decode_desc* desc, dsa_step_ring* ring,
                                const void* host_in, float* host_out, const uint8_t* k_fp8,
                                const float* k_scale, const uint16_t* kv, float sm_scale,
                                int32_t num_splits, int32_t max_seqlen, void* stream) {
  if (!desc || !ring || !host_in || !host_out || ring->step < 0) return DSA_ERR_INVALID_ARG;
  for (int b = 0; b < 2; ++b)
    if (!ring->dev_in[b] || !aligned(ring->dev_in[b], 256) || !ring->out[b] ||
        !ring->ev_in[b] || !ring->ev_done[b] || !ring->ev_out[b])
      return DSA_ERR_INVALID_ARG;
  dsa_step_layout L;
  dsa_status st = dsa_step_layout_get(desc->batch, desc->q_per_req, desc->num_heads,
                                      desc->max_pages, &L);
  if (st != DSA_OK) return st;
  const int b = static_cast<int>(ring->step & 1);
  uint8_t* in = static_cast<uint8_t*>(ring->dev_in[b]);
  dsa_decode_desc d = *desc;
  d.seqlens = reinterpret_cast<const int32_t*>(in + L.seqlens);
  d.page_table = reinterpret_cast<const int32_t*>(in + L.page_table);
  const uint8_t* q_fp8 = in + L.q_fp8;
  const float* q_scale = reinterpret_cast<const float*>(in + L.q_scale);
  const float* w = reinterpret_cast<const float*>(in + L.w);
  const uint16_t* q = reinterpret_cast<const uint16_t*>(in + L.q);
  // Both slots are checked before the first call queues anything.
  for (int s2 = 0; s2 < 2; ++s2) {
    st = fused_layer(&d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, nullptr,
                     nullptr, sm_scale, num_splits, max_seqlen, ring->out[s2], ring->ws,
                     ring->ws_bytes, stream, nullptr, /*check_only=*/true);
    if (st != DSA_OK) return st;
  }
  cudaStream_t comp = static_cast<cudaStream_t>(stream);
  cudaStream_t cin = static_cast<cudaStream_t>(ring->copy_in_stream);
  cudaStream_t cout = static_cast<cudaStream_t>(ring->copy_out_stream);
  auto ev = [](void* e) { return static_cast<cudaEvent_t>(e); };
  const bool again = ring->step >= 2;
  if (again && cudaStreamWaitEvent(cin, ev(ring->ev_done[b]), 0) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpyAsync(in, host_in, L.bytes, cudaMemcpyHostToDevice, cin) != cudaSuccess ||
      cudaEventRecord(ev(ring->ev_in[b]), cin) != cudaSuccess ||
      cudaStreamWaitEvent(comp, ev(ring->ev_in[b]), 0) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (again && cudaStreamWaitEvent(comp, ev(ring->ev_out[b]), 0) != cudaSuccess) return DSA_ERR_CUDA;
  st = fused_layer(&d, nullptr, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, nullptr, nullptr,
                   nullptr, sm_scale, num_splits, max_seqlen, ring->out[b], ring->ws,
                   ring->ws_bytes, stream, nullptr);
  if (st != DSA_OK) return st;
  const size_t ob = static_cast<size_t>(rows_of(&d)) * d.num_heads * DSA_V_DIM * sizeof(float);
  if (cudaEventRecord(ev(ring->ev_done[b]), comp) != cudaSuccess ||
      cudaStreamWaitEvent(cout, ev(ring->ev_done[b]), 0) != cudaSuccess ||
      cudaMemcpyAsync(host_out, ring->out[b], ob, cudaMemcpyDeviceToHost, cout) != cudaSuccess ||
      cudaEventRecord(ev(ring->ev_out[b]), cout) != cudaSuccess)
    return DSA_ERR_CUDA;
  ++ring->step;
  return DSA_OK;
}

dsa_status dsa_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  const int codes[5] = {dsa::fetch_error_indexer(), dsa::fetch_error_topk(), dsa::fetch_error_mla(),
                        dsa::fetch_error_merge(), dsa::fetch_error_cache()};
  for (int c : codes)
    if (c != 0) return static_cast<dsa_status>(c);
  return DSA_OK;
}

}  // extern "C"
