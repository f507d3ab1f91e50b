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
//   pass 2  topk_select_kernel, one CTA per 8192 positions of a row: finds the
//           bin b* where the count from the top crosses k, marks every
//           position above b* in the row's selection bitmap (one bit per
//           position, written without atomics: each thread owns 16
//           consecutive positions) and stores the positions in b* as
//           candidates in its chunk's own slice of the candidate list; the
//           last CTA of the row (ticket counter) resolves the candidates with
//           more radix levels over the remaining 21 key bits and, for exact
//           ties, a radix select over the position, sets the winners' bits,
//           and writes the row in ascending position order by a scan of the
//           bitmap.
#include <mutex>

#include "dsa.h"
#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(topk)

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kPer = kTopkChunk / kThreads;           // consecutive positions per thread
constexpr int kPairMax = 1024;                        // sub-candidates ranked pairwise
constexpr int kOffHist = 0;                           // 2048 x u32
constexpr int kOffCand = kOffHist + kHistBins * 4;    // kTopkChunk x uint2
constexpr int kOffSub = kOffCand + kTopkChunk * 8;    // kPairMax x uint2
constexpr int kSmemBytes = kOffSub + kPairMax * 8;    // 80 KB
static_assert(kPer == 16, "a thread pair fills one 32-bit bitmap word");

__device__ __forceinline__ int visible(const int32_t* seqlens, int t, int nq) {
  return seqlens[t / nq] - (nq - 1 - t % nq);
}

// Index of the n-th (0-based) set bit of m (m has more than n set bits).
__device__ __forceinline__ int nth_set_bit(uint32_t m, int n) {
  int pos = 0;
#pragma unroll
  for (int width = 16; width > 0; width >>= 1) {
    const uint32_t low = m & ((1u << width) - 1u);
    const int c = __popc(low);
    if (n >= c) {
      n -= c;
      m >>= width;
      pos += width;
    } else {
      m = low;
    }
  }
  return pos;
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
  uint2* scand = reinterpret_cast<uint2*>(smem + kOffCand);
  uint2* sub = reinterpret_cast<uint2*>(smem + kOffSub);
  __shared__ uint32_t scratch[40];
  __shared__ int res[2];
  __shared__ int s_info[4];   // candidates of this CTA, last flag, winners, sub count
  __shared__ int s_pref[kTopkMaxChunks + 1];

  // Everything this kernel reads may come from the kernel before it.
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.y;
  const int k = p.k;
  const int vis = visible(p.seqlens, t, p.nq);
  const int lane = threadIdx.x & 31;
  int32_t* out_row = p.out + static_cast<long long>(t) * k;

  if (vis <= k) {
    // Every visible token is selected (the short-context case).
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < k; i += kThreads) out_row[i] = i < vis ? i : -1;
    return;
  }
  const int nch = (vis + kTopkChunk - 1) / kTopkChunk;
  const int x = blockIdx.x;
  if (x >= nch) return;
  uint32_t* ctl = p.counters + static_cast<long long>(t) * topk_ctl_words(p.ld);
  uint2* cand_row = p.cand + static_cast<long long>(t) * p.ld;
  uint32_t* bm_row = p.bitmap + static_cast<long long>(t) * topk_bitmap_words(p.ld);

  // ---- this CTA's chunk: 16 consecutive scores per thread (through L1: a
  //      warp's four 16-byte loads share their cache lines), loaded before
  //      the row histogram (one latency for both).
  const float* row = p.logits + static_cast<long long>(t) * p.ld;
  const int lo = x * kTopkChunk;
  const int hi = min(vis, lo + kTopkChunk);
  const int s0 = lo + kPer * static_cast<int>(threadIdx.x);
  float v[kPer];
  if (s0 + kPer <= hi) {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + s0) + q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = s0 + j < hi ? __ldg(row + s0 + j) : 0.f;
  }
  const uint32_t* gh = p.hist + static_cast<long long>(t) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = __ldcg(gh + i);
  if (threadIdx.x == 0) s_info[0] = 0;
  __syncthreads();
  // ---- threshold bin b*: the count of scores in bins above it (nabove) is
  //      < k and reaches k with it.
  find_crossing(sh, static_cast<uint32_t>(k), true, res, scratch);
  const int bstar = res[0];
  const int nabove = res[1];
  if (bstar < 0) {  // histogram inconsistent with the row
    if (threadIdx.x == 0) raise_error(kErrCheck);
    return;
  }
  const uint32_t ub = static_cast<uint32_t>(bstar);
  uint32_t above = 0, inbin = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (s0 + j < hi) {
      const uint32_t bin = float_key(v[j]) >> kHistShift;
      if (bin > ub) above |= 1u << j;
      else if (bin == ub) inbin |= 1u << j;
    }
  }
  // Positions above b* -> the bitmap: threads 2w and 2w+1 fill word w of the
  // chunk (every word of [lo, hi) is written, so the bitmap needs no clear).
  const uint32_t upper = __shfl_down_sync(0xffffffffu, above, 1);
  if ((threadIdx.x & 1) == 0 && s0 < hi) bm_row[s0 >> 5] = above | (upper << 16);
  // Positions in b* -> this chunk's slice of the candidate list.
  const int mine = __popc(inbin);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int wbase = 0;
  if (lane == 31) wbase = atomicAdd(&s_info[0], incl);
  wbase = __shfl_sync(0xffffffffu, wbase, 31);
  {
    int pos = lo + wbase + incl - mine;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if ((inbin >> j) & 1u) cand_row[pos++] = make_uint2(float_key(v[j]), static_cast<uint32_t>(s0 + j));
  }
  // The barrier orders the block's writes before thread 0's release fence;
  // the last CTA's acquire fence then sees every CTA's writes.
  __syncthreads();
  if (threadIdx.x == 0) {
    ctl[4 + x] = static_cast<uint32_t>(s_info[0]);
    __threadfence();
    const uint32_t ticket = atomicAdd(ctl, 1u);
    const bool last = ticket == static_cast<uint32_t>(nch - 1);
    if (last) __threadfence();
    s_info[1] = last ? 1 : 0;
  }
  __syncthreads();
  if (!s_info[1]) return;

  // ---- last CTA of the row: gather the candidates of bin b*.
  {
    const uint32_t c = threadIdx.x < static_cast<unsigned>(nch) ? __ldcg(ctl + 4 + threadIdx.x) : 0u;
    const uint32_t e = block_excl_scan_512(c, scratch);
    if (threadIdx.x <= static_cast<unsigned>(nch)) s_pref[threadIdx.x] = static_cast<int>(e);
  }
  if (threadIdx.x == 0) { s_info[2] = 0; s_info[3] = 0; }
  __syncthreads();
  const int nc = s_pref[nch];
  if (static_cast<uint32_t>(nc) != sh[ub]) {   // candidates disagree with the histogram
    if (threadIdx.x == 0) raise_error(kErrCheck);
    return;
  }
  // Candidate e lives in chunk c (s_pref[c] <= e < s_pref[c + 1]).
  auto chunk_of = [&](int e) -> int {
    int a = 0, b = nch - 1;
    while (a < b) {
      const int m = (a + b + 1) >> 1;
      if (s_pref[m] <= e) a = m; else b = m - 1;
    }
    return a;
  };
  const bool in_smem = nc <= kTopkChunk;
  auto cget = [&](int e) -> uint2 {
    if (in_smem) return scand[e];
    const int c = chunk_of(e);
    return __ldcg(cand_row + static_cast<long long>(c) * kTopkChunk + (e - s_pref[c]));
  };
  if (in_smem) {
    // Four loads in flight per thread, then their four stores.
    for (int e0 = threadIdx.x; e0 < nc; e0 += 4 * kThreads) {
      uint2 cv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * kThreads;
        if (e < nc) {
          const int c = chunk_of(e);
          cv[u] = __ldcg(cand_row + static_cast<long long>(c) * kTopkChunk + (e - s_pref[c]));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u * kThreads < nc) scand[e0 + u * kThreads] = cv[u];
    }
    __syncthreads();
  }
  // A winner's bit goes into the bitmap (the CTAs that wrote it are done).
  auto take = [&](uint32_t s) {
    atomicOr(bm_row + (s >> 5), 1u << (s & 31));
    atomicAdd(&s_info[2], 1);
  };

  // ---- resolve: the need best candidates by (key desc, position asc).
  const uint32_t need = static_cast<uint32_t>(k - nabove);
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
      const uint32_t key = cget(e).x;
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
    const uint32_t hi_digits = kprefix >> 10;
    for (int e = threadIdx.x; e < nc; e += kThreads) {
      const uint2 c = cget(e);
      const uint32_t cd = c.x >> 10;
      if (cd > hi_digits) take(c.y);
      else if (cd == hi_digits) sub[atomicAdd(&s_info[3], 1)] = c;
    }
    __syncthreads();
    const int m = s_info[3];
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const uint2 ci = sub[i];
      uint32_t rank = 0;
      for (int j2 = 0; j2 < m; ++j2) {
        const uint2 cj = sub[j2];
        rank += (cj.x > ci.x || (cj.x == ci.x && cj.y < ci.y)) ? 1u : 0u;
      }
      if (rank < need_l) take(ci.y);
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
          const uint2 c = cget(e);
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
      const uint2 c = cget(e);
      if (c.x > kstar || (c.x == kstar && c.y <= istar)) take(c.y);
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0 && nabove + s_info[2] != k) raise_error(kErrCheck);

  // ---- the row in ascending position order from the bitmap, staged in
  //      shared memory (the candidate buffer) in slices of 8192 words with
  //      their exclusive bit-count prefix.  Output j is then found by a
  //      binary search over the prefix, so every thread writes about k / 512
  //      outputs however the selected bits cluster.
  const int nwords = (vis + 31) >> 5;
  uint32_t* sbm = reinterpret_cast<uint32_t*>(smem + kOffCand);
  constexpr int kSlice = kTopkChunk;       // words: bitmap + prefix = the 64 KB buffer
  uint32_t* spre = sbm + kSlice;
  uint32_t base = 0;
  for (int c0 = 0; c0 < nwords; c0 += kSlice) {
    const int cn = min(kSlice, nwords - c0);
    __syncthreads();   // the previous slice (or the candidates) is no longer read
    for (int i = threadIdx.x; i < cn; i += kThreads) sbm[i] = __ldcg(bm_row + c0 + i);
    __syncthreads();
    const int per = (cn + kThreads - 1) / kThreads;
    const int w0 = min(cn, static_cast<int>(threadIdx.x) * per), w1 = min(cn, w0 + per);
    uint32_t cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(sbm[w]);
    uint32_t run = block_excl_scan_512(cnt, scratch);
    const uint32_t total = scratch[16 + 15];   // inclusive sum over the block
    for (int w = w0; w < w1; ++w) {
      spre[w] = run;
      run += __popc(sbm[w]);
    }
    __syncthreads();
    for (uint32_t j = threadIdx.x; j < total; j += kThreads) {
      int a = 0, b = cn - 1;   // the last word whose prefix is <= j holds output j
      while (a < b) {
        const int m = (a + b + 1) >> 1;
        if (spre[m] <= j) a = m; else b = m - 1;
      }
      if (base + j < static_cast<uint32_t>(k))
        out_row[base + j] = (c0 + a) * 32 + nth_set_bit(sbm[a], static_cast<int>(j - spre[a]));
    }
    base += total;
  }
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) {
  const int T = a.batch * a.nq;
  const int chunks = static_cast<int>((a.ld + kTopkChunk - 1) / kTopkChunk);
  if (chunks > kTopkMaxChunks) return cudaErrorInvalidValue;
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
                       a.pdl != 0 && a.hist_ready, 1, a);
}

// ---------------------------------------------------------------------------
// Top-k without a caller-provided workspace (dsa_topk_noalloc).
//
// For callers that cannot allocate device memory at the point where they run
// the selection, the histogram, control words, candidate lists and selection
// bitmap live in one statically sized device array.  Every GPU that loads the library reserves
// it (kNoAllocScratchBytes) until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxRows = 64;                 // query rows T
constexpr long long kNoAllocMaxScores = 1ll << 21;  // T * ld_logits
constexpr size_t kNoAllocHistBytes = size_t(kNoAllocMaxRows) * kHistBins * 4;
constexpr size_t kNoAllocCounterOff = kNoAllocHistBytes;
// Control words: 4 per row plus one per 8192-score chunk, over all rows at
// most 4 T + T + 2^21 / 8192 words.
constexpr size_t kNoAllocCounterWords =
    size_t(kNoAllocMaxRows) * 5 + size_t(kNoAllocMaxScores) / kTopkChunk;
constexpr size_t kNoAllocCandOff =
    (kNoAllocCounterOff + kNoAllocCounterWords * 4 + 255) & ~size_t(255);
constexpr size_t kNoAllocBitmapOff = kNoAllocCandOff + size_t(kNoAllocMaxScores) * 8;
// Bitmap: ceil(ld / 32) words per row, at most 2^21 / 32 + T words.
constexpr size_t kNoAllocScratchBytes =
    kNoAllocBitmapOff + (size_t(kNoAllocMaxScores) / 32 + kNoAllocMaxRows) * 4;

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
  a.bitmap = reinterpret_cast<uint32_t*>(base + kNoAllocBitmapOff);
  a.batch = d->batch; a.nq = d->q_per_req; a.k = d->topk; a.hist_ready = 0;
  return launch_topk(a, s) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
