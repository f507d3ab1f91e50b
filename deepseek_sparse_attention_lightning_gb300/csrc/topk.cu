// topk.cu -- stage 2, per-query top-k without a sort.
//
// Each query row t keeps the n = min(k, vis[t]) visible positions with the
// largest fp32 score; equal scores go to the lower position ("MTP and sparse
// attention: NSA and DSA", section "Sparse attention: NSA and DSA": each query
// keeps its 2048 highest-scoring tokens).  The selection is exact.
//
// Scores are compared through an order-preserving 32-bit key (-0 == +0).
//   pass 1  histogram of the top 11 key bits per row (fused into the indexer
//           epilogue on the fused path, else topk_hist_kernel);
//   pass 2  topk_select_kernel, many CTAs per row: finds the bin b* where the
//           count from the top crosses k, writes every position above b*
//           straight to the output and appends the positions in b* to a
//           candidate list; the last CTA of the row (ticket counter) resolves
//           the candidates with two more radix levels over the remaining 21
//           key bits and, for exact ties, a radix select over the position,
//           then rewrites the row in ascending position order through a
//           shared-memory bitmap.
#include <mutex>

#include "dsa.h"
#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(topk)

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kSelMax = 2048;                         // positions above b* per chunk < k
constexpr int kPairMax = 1024;                        // sub-candidates ranked pairwise (fit in ssel)
constexpr int kOffHist = 0;                           // 2048 x u32
constexpr int kOffSel = kOffHist + kHistBins * 4;     // 2048 x i32
constexpr int kOffCand = kOffSel + kSelMax * 4;       // kTopkChunk x uint2
constexpr int kSmemBytes = kOffCand + kTopkChunk * 8; // 80 KB, reused as the bitmap
constexpr int kBitmapWords = kSmemBytes / 4;

__device__ __forceinline__ int visible(const int32_t* seqlens, int t, int nq) {
  return seqlens[t / nq] - (nq - 1 - t % nq);
}

// Cache row of logical position s of request r (-1 if its page id is bad).
__device__ __forceinline__ int phys_row(const TopkLaunch& p, int r, int s) {
  const int pg = p.page_table[static_cast<long long>(r) * p.max_pages + (s >> 6)];
  if (pg < 0 || pg >= p.num_pages) {
    raise_error(kErrCheck);
    return -1;
  }
  return pg * kPage + (s & (kPage - 1));
}

// Exclusive scan of one value per thread over a 512-thread block.
__device__ __forceinline__ uint32_t block_excl_scan_512(uint32_t v, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < 16 ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < 16) scratch[16 + lane] = w;
  }
  __syncthreads();
  const uint32_t off = warp ? scratch[16 + warp - 1] : 0u;
  return off + x - v;
}

// Over bins h[0..2048): the bin where the running count, taken from the top
// bin down (descending) or from bin 0 up, first reaches `need` (>= 1).
// res[0] = that bin (-1 if none), res[1] = the count strictly before it.
__device__ void find_crossing(const uint32_t* h, uint32_t need, bool descending, int* res,
                              uint32_t* scratch) {
  uint32_t c[4], local = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int b = descending ? (kHistBins - 1 - 4 * threadIdx.x - e) : (4 * threadIdx.x + e);
    c[e] = h[b];
    local += c[e];
  }
  if (threadIdx.x == 0) res[0] = -1;
  const uint32_t excl = block_excl_scan_512(local, scratch);
  if (excl < need && excl + local >= need) {
    uint32_t run = excl;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int b = descending ? (kHistBins - 1 - 4 * threadIdx.x - e) : (4 * threadIdx.x + e);
      if (run + c[e] >= need) {
        res[0] = b;
        res[1] = static_cast<int>(run);
        break;
      }
      run += c[e];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
    topk_hist_kernel(const TopkLaunch p) {
  __shared__ uint32_t sh[kHistBins];
  const int t = blockIdx.y;
  const int vis = visible(p.seqlens, t, p.nq);
  const int lo = blockIdx.x * kTopkChunk;
  if (vis <= p.k || lo >= vis) return;
  const int hi = min(vis, lo + kTopkChunk);
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = 0u;
  __syncthreads();
  const float* row = p.logits + static_cast<long long>(t) * p.ld;
  const int vend = lo + ((hi - lo) & ~3);
  for (int s = lo + 4 * threadIdx.x; s < vend; s += 4 * kThreads) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row + s));
    atomicAdd(&sh[float_key(v.x) >> kHistShift], 1u);
    atomicAdd(&sh[float_key(v.y) >> kHistShift], 1u);
    atomicAdd(&sh[float_key(v.z) >> kHistShift], 1u);
    atomicAdd(&sh[float_key(v.w) >> kHistShift], 1u);
  }
  for (int s = vend + threadIdx.x; s < hi; s += kThreads)
    atomicAdd(&sh[float_key(__ldg(row + s)) >> kHistShift], 1u);
  __syncthreads();
  uint32_t* gh = p.hist + static_cast<long long>(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads)
    if (sh[i]) atomicAdd(gh + i, sh[i]);
}

__global__ void __launch_bounds__(kThreads)
    topk_select_kernel(const TopkLaunch p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* sh = reinterpret_cast<uint32_t*>(smem + kOffHist);
  int* ssel = reinterpret_cast<int*>(smem + kOffSel);
  uint2* scand = reinterpret_cast<uint2*>(smem + kOffCand);
  __shared__ uint32_t scratch[40];
  __shared__ int res[2];
  __shared__ int s_info[8];   // nsel, ncand, base, cbase, last, emit, sub count

  // Everything this kernel reads may come from the kernel before it.
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.y;
  const int k = p.k;
  const int vis = visible(p.seqlens, t, p.nq);
  int32_t* out_row = p.out + static_cast<long long>(t) * k;

  const int req = t / p.nq;
  if (vis <= k) {
    // Every visible token is selected (the short-context case).
    if (blockIdx.x == 0) {
      int32_t* rows_row = p.rows ? p.rows + static_cast<long long>(t) * k : nullptr;
      for (int i = threadIdx.x; i < k; i += kThreads) {
        out_row[i] = i < vis ? i : -1;
        if (rows_row) {
          const int row = i < vis ? phys_row(p, req, i) : -1;
          rows_row[i] = row;
        }
      }
    }
    return;
  }
  const int nch = (vis + kTopkChunk - 1) / kTopkChunk;
  if (static_cast<int>(blockIdx.x) >= nch) return;
  uint32_t* counters = p.counters + static_cast<long long>(t) * kCounterWords;
  uint2* cand_row = p.cand + static_cast<long long>(t) * p.ld;

  // ---- this CTA's chunk of the row: all of a thread's scores are loaded
  //      first (one latency), then the row histogram.
  const float* row = p.logits + static_cast<long long>(t) * p.ld;
  const int lo = blockIdx.x * kTopkChunk;
  const int hi = min(vis, lo + kTopkChunk);
  constexpr int kIters = kTopkChunk / (4 * kThreads);
  float x[kIters][4];
#pragma unroll
  for (int q = 0; q < kIters; ++q) {
    const int s = lo + q * 4 * kThreads + 4 * static_cast<int>(threadIdx.x);
    if (s + 3 < hi) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(row + s));
      x[q][0] = v.x; x[q][1] = v.y; x[q][2] = v.z; x[q][3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[q][e] = s + e < hi ? __ldcg(row + s + e) : 0.f;
    }
  }
  // ---- threshold bin b*: the count of scores in bins above it is < k and
  //      reaches k with it.
  const uint32_t* gh = p.hist + static_cast<long long>(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = __ldcg(gh + i);
  __syncthreads();
  find_crossing(sh, static_cast<uint32_t>(k), true, res, scratch);
  const int bstar = res[0];
  if (bstar < 0) {  // histogram inconsistent with the row
    if (threadIdx.x == 0) raise_error(kErrCheck);
    return;
  }
  const uint32_t ub = static_cast<uint32_t>(bstar);
  // Classify the thread's scores, then place them with one block scan of the
  // packed (candidates << 16 | selected) counts.
  uint32_t above = 0, inbin = 0;
#pragma unroll
  for (int q = 0; q < kIters; ++q) {
    const int s = lo + q * 4 * kThreads + 4 * static_cast<int>(threadIdx.x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t bin = float_key(x[q][e]) >> kHistShift;
      const uint32_t bit = 1u << (4 * q + e);
      if (s + e < hi) {
        if (bin > ub) above |= bit;
        else if (bin == ub) inbin |= bit;
      }
    }
  }
  const uint32_t mine = (static_cast<uint32_t>(__popc(inbin)) << 16) | __popc(above);
  const uint32_t off = block_excl_scan_512(mine, scratch);
  if (threadIdx.x == kThreads - 1) {
    s_info[0] = static_cast<int>((off + mine) & 0xFFFFu);
    s_info[1] = static_cast<int>((off + mine) >> 16);
  }
  {
    int oa = static_cast<int>(off & 0xFFFFu), oc = static_cast<int>(off >> 16);
#pragma unroll
    for (int q = 0; q < kIters; ++q) {
      const int s = lo + q * 4 * kThreads + 4 * static_cast<int>(threadIdx.x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bit = 1u << (4 * q + e);
        if (above & bit) {
          if (oa < kSelMax) ssel[oa] = s + e;
          ++oa;
        } else if (inbin & bit) {
          scand[oc++] = make_uint2(float_key(x[q][e]), static_cast<uint32_t>(s + e));
        }
      }
    }
  }
  __syncthreads();
  const int nsel = s_info[0], ncand = s_info[1];
  if (threadIdx.x == 0) {
    if (nsel > kSelMax) raise_error(kErrCheck);
    // One 64-bit atomic reserves room in both lists: (candidates, selected).
    const unsigned long long add =
        (static_cast<unsigned long long>(ncand) << 32) | static_cast<unsigned long long>(nsel);
    const unsigned long long old =
        atomicAdd(reinterpret_cast<unsigned long long*>(counters), add);
    s_info[2] = static_cast<int>(old & 0xFFFFFFFFull);
    s_info[3] = static_cast<int>(old >> 32);
  }
  __syncthreads();
  {
    const int base = s_info[2], cbase = s_info[3];
    const int nw = min(nsel, kSelMax);
    for (int i = threadIdx.x; i < nw; i += kThreads)
      if (base + i < k) out_row[base + i] = ssel[i];
    for (int i = threadIdx.x; i < ncand; i += kThreads) cand_row[cbase + i] = scand[i];
  }
  // The barrier orders the block's writes before thread 0's release fence;
  // the last CTA's acquire fence then sees every CTA's writes.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t ticket = atomicAdd(counters + 2, 1u);
    const bool last = ticket == static_cast<uint32_t>(nch - 1);
    if (last) __threadfence();
    s_info[4] = last ? 1 : 0;
  }
  __syncthreads();
  if (!s_info[4]) return;

  // ---- last CTA of the row: resolve the candidates of bin b*.
  const int nabove = static_cast<int>(__ldcg(counters + 0));
  const int nc = static_cast<int>(__ldcg(counters + 1));
  const uint32_t need = static_cast<uint32_t>(k - nabove);
  const uint2* cp = cand_row;
  if (nc <= kTopkChunk) {
    for (int i = threadIdx.x; i < nc; i += kThreads) scand[i] = __ldcg(cand_row + i);
    cp = scand;
  }
  if (threadIdx.x == 0) s_info[5] = 0;
  __syncthreads();

  uint32_t kprefix = ub << kHistShift, kmask = 0xFFFFFFFFu << kHistShift;
  uint32_t need_l = need;
  uint32_t cnt_eq = 0;
  const int kshift[2] = {10, 0};
  const int kwidth[2] = {11, 10};
  bool ok = need >= 1;
  bool pairwise = false;
  for (int lvl = 0; lvl < 2 && ok; ++lvl) {
    const int sh_ = kshift[lvl];
    const uint32_t dm = (1u << kwidth[lvl]) - 1u;
    for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = 0u;
    __syncthreads();
    for (int e = threadIdx.x; e < nc; e += kThreads) {
      const uint32_t key = cp[e].x;
      if ((key & kmask) == kprefix) atomicAdd(&sh[(key >> sh_) & dm], 1u);
    }
    __syncthreads();
    find_crossing(sh, need_l, true, res, scratch);
    if (res[0] < 0) { ok = false; break; }
    const uint32_t d = static_cast<uint32_t>(res[0]);
    cnt_eq = sh[d];
    need_l -= static_cast<uint32_t>(res[1]);
    kprefix |= d << sh_;
    kmask |= dm << sh_;
    __syncthreads();
    // Few candidates left in the crossing digit: rank them pairwise instead
    // of further radix levels.
    if (lvl == 0 && cnt_eq <= static_cast<uint32_t>(kPairMax)) {
      pairwise = true;
      break;
    }
  }
  if (!ok) {
    if (threadIdx.x == 0) raise_error(kErrCheck);
    return;
  }
  if (pairwise) {
    // Candidates whose digit is above the crossing one are in; of those with
    // the crossing digit (m <= kPairMax), the need_l best by (key desc,
    // position asc) are in.
    uint2* sub = reinterpret_cast<uint2*>(ssel);
    if (threadIdx.x == 0) s_info[6] = 0;
    __syncthreads();
    const uint32_t hi_digits = kprefix >> 10;
    for (int e = threadIdx.x; e < nc; e += kThreads) {
      const uint2 c = cp[e];
      const uint32_t cd = c.x >> 10;
      if (cd > hi_digits) {
        const int pos = atomicAdd(&s_info[5], 1);
        if (nabove + pos < k) out_row[nabove + pos] = static_cast<int>(c.y);
      } else if (cd == hi_digits) {
        sub[atomicAdd(&s_info[6], 1)] = c;
      }
    }
    __syncthreads();
    const int m = s_info[6];
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const uint2 ci = sub[i];
      uint32_t rank = 0;
      for (int j2 = 0; j2 < m; ++j2) {
        const uint2 cj = sub[j2];
        rank += (cj.x > ci.x || (cj.x == ci.x && cj.y < ci.y)) ? 1u : 0u;
      }
      if (rank < need_l) {
        const int pos = atomicAdd(&s_info[5], 1);
        if (nabove + pos < k) out_row[nabove + pos] = static_cast<int>(ci.y);
      }
    }
  } else {
    const uint32_t kstar = kprefix;
    // Exact ties at the threshold key: keep the need_l lowest positions.
    uint32_t istar = 0xFFFFFFFFu;
    if (need_l < cnt_eq) {
      uint32_t iprefix = 0, imask = 0, need_i = need_l;
      const int ishift[3] = {20, 10, 0};
      const int iwidth[3] = {11, 10, 10};
      for (int lvl = 0; lvl < 3 && ok; ++lvl) {
        const int sh_ = ishift[lvl];
        const uint32_t dm = (1u << iwidth[lvl]) - 1u;
        for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = 0u;
        __syncthreads();
        for (int e = threadIdx.x; e < nc; e += kThreads) {
          const uint2 c = cp[e];
          if (c.x == kstar && (c.y & imask) == iprefix) atomicAdd(&sh[(c.y >> sh_) & dm], 1u);
        }
        __syncthreads();
        find_crossing(sh, need_i, false, res, scratch);
        if (res[0] < 0) { ok = false; break; }
        need_i -= static_cast<uint32_t>(res[1]);
        iprefix |= static_cast<uint32_t>(res[0]) << sh_;
        imask |= dm << sh_;
        __syncthreads();
      }
      istar = iprefix;
    }
    if (!ok) {
      if (threadIdx.x == 0) raise_error(kErrCheck);
      return;
    }
    for (int e = threadIdx.x; e < nc; e += kThreads) {
      const uint2 c = cp[e];
      if (c.x > kstar || (c.x == kstar && c.y <= istar)) {
        const int pos = atomicAdd(&s_info[5], 1);
        if (nabove + pos < k) out_row[nabove + pos] = static_cast<int>(c.y);
      }
    }
  }
  __threadfence_block();
  __syncthreads();
  if (threadIdx.x == 0 && nabove + s_info[5] != k) raise_error(kErrCheck);

  // ---- rewrite the row in ascending position order through a bitmap.
  const int nwords = (vis + 31) >> 5;
  if (nwords <= kBitmapWords) {
    uint32_t* bm = reinterpret_cast<uint32_t*>(smem);
    for (int i = threadIdx.x; i < nwords; i += kThreads) bm[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += kThreads) {
      const int s = __ldcg(out_row + i);
      if (s >= 0 && s < vis) atomicOr(&bm[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    const int per = (nwords + kThreads - 1) / kThreads;
    const int w0 = min(nwords, threadIdx.x * per), w1 = min(nwords, w0 + per);
    uint32_t cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
    uint32_t pos = block_excl_scan_512(cnt, scratch);
    for (int w = w0; w < w1; ++w) {
      uint32_t bits = bm[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < static_cast<uint32_t>(k)) out_row[pos] = w * 32 + b;
        ++pos;
      }
    }
  }
  if (p.rows) {
    // Fused index -> cache-row transform of the final selection.
    __syncthreads();
    int32_t* rows_row = p.rows + static_cast<long long>(t) * k;
    for (int i = threadIdx.x; i < k; i += kThreads) {
      const int s = __ldcg(out_row + i);
      rows_row[i] = (s >= 0 && s < vis) ? phys_row(p, req, s) : -1;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) {
  const int T = a.batch * a.nq;
  const int chunks = static_cast<int>((a.ld + kTopkChunk - 1) / kTopkChunk);
  dim3 grid(chunks > 0 ? chunks : 1, T);
  if (!a.hist_ready) {
    topk_hist_kernel<<<grid, kThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_kernel(topk_select_kernel, grid, dim3(kThreads), kSmemBytes, stream,
                       a.pdl != 0 && a.hist_ready, a);
}

// ---------------------------------------------------------------------------
// Top-k without a caller-provided workspace (dsa_topk_noalloc).
//
// For callers that cannot allocate device memory at the point where they run
// the selection, the histogram, counters and candidate lists live in one
// statically sized device array.  Every GPU that loads the library reserves
// it (kNoAllocScratchBytes) until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxRows = 64;                 // query rows T
constexpr long long kNoAllocMaxScores = 1ll << 21;  // T * ld_logits
constexpr size_t kNoAllocHistBytes = size_t(kNoAllocMaxRows) * kHistBins * 4;
constexpr size_t kNoAllocCounterOff = kNoAllocHistBytes;
constexpr size_t kNoAllocCandOff =
    (kNoAllocCounterOff + size_t(kNoAllocMaxRows) * kCounterWords * 4 + 255) & ~size_t(255);
constexpr size_t kNoAllocScratchBytes = kNoAllocCandOff + size_t(kNoAllocMaxScores) * 8;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device; the host-side symbol is not a device address).
void* noalloc_scratch(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = ptr;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_topk_noalloc(const dsa_decode_desc* d, const float* logits,
                                       int64_t ld, int32_t* topk_idx, void* stream) {
  using namespace dsa;
  if (!d || d->batch < 1 || d->q_per_req < 1 || d->num_heads < 1 || d->topk < 1 ||
      d->max_pages < 1 || d->num_pages < 1 || !d->seqlens || !d->page_table)
    return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(d->seqlens) & 3) || (reinterpret_cast<uintptr_t>(d->page_table) & 3))
    return DSA_ERR_INVALID_ARG;
  if (d->batch > DSA_MAX_BATCH || d->q_per_req > DSA_MAX_Q_PER_REQ || d->topk > DSA_MAX_TOPK ||
      d->page_size != DSA_PAGE_SIZE)
    return DSA_ERR_UNSUPPORTED;
  if (!logits || !topk_idx || (reinterpret_cast<uintptr_t>(logits) & 15) ||
      (reinterpret_cast<uintptr_t>(topk_idx) & 3))
    return DSA_ERR_INVALID_ARG;
  if (ld < static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE || ld % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  const int T = d->batch * d->q_per_req;
  if (T > kNoAllocMaxRows || static_cast<long long>(T) * ld > kNoAllocMaxScores)
    return DSA_ERR_UNSUPPORTED;   // beyond the fixed scratch: use dsa_topk with a workspace
  cudaError_t e;
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch(&e));
  if (!base) return DSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The previous call's histogram and counters are still there: clear them.
  e = cudaMemsetAsync(base, 0, kNoAllocCandOff, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  TopkLaunch a{};
  a.seqlens = d->seqlens; a.logits = logits; a.ld = ld; a.out = topk_idx;
  a.hist = reinterpret_cast<uint32_t*>(base);
  a.counters = reinterpret_cast<uint32_t*>(base + kNoAllocCounterOff);
  a.cand = reinterpret_cast<uint2*>(base + kNoAllocCandOff);
  a.batch = d->batch; a.nq = d->q_per_req; a.k = d->topk; a.hist_ready = 0;
  return launch_topk(a, s) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
