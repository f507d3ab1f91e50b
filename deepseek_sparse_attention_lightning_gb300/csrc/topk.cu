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
//   pass 2  topk_select_kernel: each row is one cluster of 16 CTAs, CTA x
//           owning chunk x of the row (8192, 16384 or 32768 positions; a
//           warp's score loads are 512 consecutive bytes).  Every CTA finds
//           the bin b* where the count from the top crosses k, marks the
//           positions above b* in its shared-memory slice of the selection
//           bitmap and keeps the positions in b* as candidates in its own
//           shared memory (the rare excess over 512 in a global list).  After
//           a cluster barrier, CTA 0 reads every CTA's candidates through
//           distributed shared memory and resolves them with more radix
//           levels over the remaining 21 key bits (a pairwise rank once few
//           are left, a radix select over the position for exact ties) into
//           one threshold (key, position): a candidate is in iff its key is
//           larger, or equal with a position not larger.  After a second
//           barrier every CTA marks its own winners, the CTAs exchange their
//           selected counts through distributed shared memory, and each
//           writes its chunk's positions, ascending, at its offset in the row.
#include <algorithm>
#include <mutex>

#include "dsa.h"
#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(topk)

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kPairMax = 128;                         // sub-candidates ranked pairwise
constexpr int kOffHist = 0;                           // 2048 x u32: the row histogram
constexpr int kOffLvl = kOffHist + kHistBins * 4;     // 2048 x u32: (CTA 0) first resolve level
constexpr int kCandSlot = kTopkChunk / 16;            // candidates per chunk kept in shared memory
static_assert(kCandSlot == kThreads, "one candidate slot per thread");
constexpr int kOffCand = kOffLvl + kHistBins * 4;     // kCandSlot x uint2: this chunk's candidates
constexpr int kOffSub = kOffCand + kCandSlot * 8;     // kPairMax x uint2
constexpr int kOffBits = kOffSub + kPairMax * 8;      // this chunk's bitmap words
constexpr int kMaxChunkMul = 4;                       // chunk = 8192 x {1, 2, 4}
constexpr int kSmemBytes = kOffBits + (kTopkChunk * kMaxChunkMul / 32) * 4;   // 25 KB

__device__ __forceinline__ int visible(const int32_t* seqlens, int t, int nq) {
  return seqlens[t / nq] - (nq - 1 - t % nq);
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

// One cluster of gridDim.x (<= kTopkClusterCtas) CTAs per query row, as many
// as the longest row needs chunks; CTA x owns chunk x of C = 512 * 4 * Q
// positions, 4 Q per thread (Q float4 loads).
template <int Q>
__global__ void __launch_bounds__(kThreads)
    topk_select_kernel(const TopkLaunch p) {
  constexpr int P = 4 * Q;             // positions per thread
  constexpr int C = kThreads * P;      // positions per CTA
  constexpr int HW = (Q + 3) / 4;      // 16-bit candidate masks per thread (4 float4 groups each)
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* sh = reinterpret_cast<uint32_t*>(smem + kOffHist);
  uint32_t* slv = reinterpret_cast<uint32_t*>(smem + kOffLvl);
  uint2* scand = reinterpret_cast<uint2*>(smem + kOffCand);
  uint2* sub = reinterpret_cast<uint2*>(smem + kOffSub);
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + kOffBits);
  __shared__ uint32_t scratch[40];
  __shared__ int res[2];
  __shared__ int s_info[4];   // candidates of this CTA, (CTA 0) all candidates, overflow, sub count
  __shared__ uint32_t s_thr[2];   // the threshold (key, position), pushed by CTA 0
  __shared__ uint32_t s_allsel[kTopkClusterCtas];   // every chunk's selected count, pushed by each
  __shared__ uint32_t s_ccnt[kTopkClusterCtas];   // (CTA 0) every chunk's candidate count, pushed by each

  // seqlens is an input of the layer that no kernel before writes: its load
  // is issued before the wait, so the score loads can follow it at once.
  // Everything else this kernel reads may come from the kernel before it.
  const int t = blockIdx.y;
  const int k = p.k;
  const int vis = visible(p.seqlens, t, p.nq);
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  int32_t* out_row = p.out + static_cast<long long>(t) * k;

  if (vis <= k) {
    // Every visible token is selected (the short-context case); the whole
    // cluster of the row leaves here.
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < k; i += kThreads) out_row[i] = i < vis ? i : -1;
    return;
  }
  const int x = static_cast<int>(cluster_ctarank());
  const int cs = static_cast<int>(gridDim.x);   // CTAs of the row's cluster
  const int nch = (vis + C - 1) / C;   // <= cs (the host sizes the cluster)
  const bool has = x < nch;
  uint2* cand_row = p.cand + static_cast<long long>(t) * p.ld;
  const int lo = x * C;
  const int hi = has ? min(vis, lo + C) : lo;

  // ---- scores: this thread's float4 f = threadIdx.x + kThreads * q holds
  //      positions lo + 4 f .. lo + 4 f + 3, so a warp's loads are 512
  //      consecutive bytes (four whole cache lines per instruction).
  const float* row = p.logits + static_cast<long long>(t) * p.ld;
  auto pos_of = [&](int q) { return lo + 4 * (static_cast<int>(threadIdx.x) + kThreads * q); };
  float v[P];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int pq = pos_of(q);
    if (pq + 4 <= hi) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + pq));
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) v[4 * q + b] = pq + b < hi ? __ldg(row + pq + b) : 0.f;
    }
  }
  if (x == 0)   // the first resolve level's histogram, ready before it is needed
    for (int i = threadIdx.x; i < kHistBins; i += kThreads) slv[i] = 0u;
  // The histogram's four words per thread are all in flight before any is
  // stored (one round trip instead of four).
  const uint32_t* gh = p.hist + static_cast<long long>(t) * kHistBins;
  {
    uint32_t hv[kHistBins / kThreads];
#pragma unroll
    for (int u = 0; u < kHistBins / kThreads; ++u) hv[u] = __ldcg(gh + threadIdx.x + u * kThreads);
#pragma unroll
    for (int u = 0; u < kHistBins / kThreads; ++u) sh[threadIdx.x + u * kThreads] = hv[u];
  }
  if (threadIdx.x == 0) s_info[0] = 0;
  __syncthreads();
  // ---- threshold bin b*: the count of scores in bins above it (nabove) is
  //      < k and reaches k with it.  Every CTA gets the same answer.
  find_crossing(sh, static_cast<uint32_t>(k), true, res, scratch);
  const int bstar = res[0];
  const int nabove = res[1];
  if (bstar < 0) {  // histogram inconsistent with the row (the whole cluster leaves)
    if (threadIdx.x == 0) raise_error(kErrCheck);
    return;
  }
  const uint32_t ub = static_cast<uint32_t>(bstar);
  // ---- classify: positions above b* -> this chunk's bitmap words, those in
  //      b* -> candidates.  Bit 4 (q mod 4) + b of inbin[q / 4] is position
  //      pos_of(q) + b.  Bitmap word 64 q + threadIdx.x / 8 holds the nibbles
  //      of eight consecutive threads (four positions each).
  uint32_t inbin[HW];
#pragma unroll
  for (int h = 0; h < HW; ++h) inbin[h] = 0u;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int pq = pos_of(q);
    uint32_t above = 0, in = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (pq + b < hi) {
        const uint32_t bin = float_key(v[4 * q + b]) >> kHistShift;
        if (bin > ub) above |= 1u << b;
        else if (bin == ub) in |= 1u << b;
      }
    inbin[q >> 2] |= in << (4 * (q & 3));
    uint32_t w = above << (4 * (lane & 7));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    w |= __shfl_xor_sync(0xffffffffu, w, 4);
    if ((lane & 7) == 0) sbits[64 * q + (threadIdx.x >> 3)] = w;
  }
  int mine = 0;
#pragma unroll
  for (int h = 0; h < HW; ++h) mine += __popc(inbin[h]);
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
    // Candidate i of this chunk goes to its slot i of this CTA's shared
    // memory if i < kCandSlot (CTA 0 reads the slots through distributed
    // shared memory after the barrier), else to the chunk's global slice.
    int i = wbase + incl - mine;
#pragma unroll
    for (int h = 0; h < HW; ++h)
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (4 * h + (j >> 2) < Q && ((inbin[h] >> j) & 1u)) {
          const int q = 4 * h + (j >> 2), b = j & 3;
          const uint2 c = make_uint2(float_key(v[4 * q + b]), static_cast<uint32_t>(pos_of(q) + b));
          if (i < kCandSlot) scand[i] = c;
          else cand_row[lo + i] = c;
          ++i;
        }
  }
  __syncthreads();
  if (threadIdx.x == 0)
    st_shared_cluster_u32(mapa_shared(smem_u32(&s_ccnt[x]), 0), has ? static_cast<uint32_t>(s_info[0]) : 0u);
  cluster_sync();   // #1: every chunk's candidates and count are in place

  // ---- CTA 0 resolves the candidates of bin b* into the threshold.
  if (x == 0) {
    if (threadIdx.x < 32) {
      // All candidates of the row, and whether a chunk overflowed its slots.
      const uint32_t c = threadIdx.x < static_cast<unsigned>(nch) ? s_ccnt[threadIdx.x] : 0u;
      uint32_t tot = c, mx = c;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (threadIdx.x == 0) {
        s_info[1] = static_cast<int>(tot);
        s_info[2] = mx > static_cast<uint32_t>(kCandSlot) ? 1 : 0;
        s_info[3] = 0;
        s_thr[0] = 0xFFFFFFFFu;   // selects no candidate (error fallback)
        s_thr[1] = 0u;
      }
    }
    __syncthreads();
    const int nc = s_info[1];
    const bool over = s_info[2] != 0;
    bool ok = static_cast<uint32_t>(nc) == sh[ub];   // candidates agree with the histogram
    // Candidates past a chunk's slots, from its global slice (rare).
    auto for_each_overflow = [&](auto&& f) {
      if (!over) return;
      for (int cx = 0; cx < nch; ++cx)
        for (int i = kCandSlot + static_cast<int>(threadIdx.x); i < static_cast<int>(s_ccnt[cx]);
             i += kThreads)
          f(__ldcg(cand_row + static_cast<long long>(cx) * C + i));
    };
    // This thread's slot of every chunk, read from the chunk's CTA: the keys
    // stay in registers for the histogram and collection passes (loaded
    // together, not one per pass behind the previous pass's atomics).
    const uint32_t slot = smem_u32(scand) + 8u * threadIdx.x;
    uint32_t ck[kTopkClusterCtas];
    uint32_t cvalid = 0;
#pragma unroll
    for (int cx = 0; cx < kTopkClusterCtas; ++cx) {
      const bool in = cx < nch && threadIdx.x < s_ccnt[cx];
      ck[cx] = in ? ld_shared_cluster_u32(mapa_shared(slot, cx)) : 0u;
      cvalid |= (in ? 1u : 0u) << cx;
    }
    // Every candidate once (the slots, then the overflow).
    auto for_each_cand = [&](auto&& f) {
      for (int cx = 0; cx < nch; ++cx)
        if (threadIdx.x < s_ccnt[cx]) {
          const uint32_t a = mapa_shared(slot, cx);
          f(make_uint2(ld_shared_cluster_u32(a), ld_shared_cluster_u32(a + 4)));
        }
      for_each_overflow(f);
    };
    // The need best candidates by (key desc, position asc).
    const uint32_t need = static_cast<uint32_t>(k - nabove);
    uint32_t kprefix = ub << kHistShift, kmask = 0xFFFFFFFFu << kHistShift;
    uint32_t need_l = need;
    uint32_t cnt_eq = 0;
    const int kshift[2] = {10, 0};
    const int kwidth[2] = {11, 10};
    ok = ok && need >= 1;
    bool pairwise = false;
    for (int lvl = 0; lvl < 2 && ok; ++lvl) {
      const int sh_ = kshift[lvl];
      const uint32_t dm = (1u << kwidth[lvl]) - 1u;
      // Level 0 counts into its own array (zeroed at the start); level 1
      // reuses the row histogram's, no longer needed.
      uint32_t* hl = lvl == 0 ? slv : sh;
      if (lvl > 0) {
        for (int i = threadIdx.x; i < kHistBins; i += kThreads) sh[i] = 0u;
        __syncthreads();
      }
#pragma unroll
      for (int cx = 0; cx < kTopkClusterCtas; ++cx)
        if (((cvalid >> cx) & 1u) && (ck[cx] & kmask) == kprefix)
          atomicAdd(&hl[(ck[cx] >> sh_) & dm], 1u);
      for_each_overflow([&](uint2 c) {
        if ((c.x & kmask) == kprefix) atomicAdd(&hl[(c.x >> sh_) & dm], 1u);
      });
      __syncthreads();
      find_crossing(hl, need_l, true, res, scratch);
      if (res[0] < 0) { ok = false; break; }
      const uint32_t d = static_cast<uint32_t>(res[0]);
      cnt_eq = hl[d];
      need_l -= static_cast<uint32_t>(res[1]);
      kprefix |= d << sh_;
      kmask |= dm << sh_;
      __syncthreads();
      if (lvl == 0 && cnt_eq <= static_cast<uint32_t>(kPairMax)) {
        pairwise = true;
        break;
      }
    }
    if (ok && pairwise) {
      // Of the candidates with the crossing digit (m <= kPairMax), the
      // need_l-th best by (key desc, position asc) is the threshold.
      const uint32_t hi_digits = kprefix >> 10;
#pragma unroll
      for (int cx = 0; cx < kTopkClusterCtas; ++cx)
        if (((cvalid >> cx) & 1u) && (ck[cx] >> 10) == hi_digits)
          sub[atomicAdd(&s_info[3], 1)] =
              make_uint2(ck[cx], ld_shared_cluster_u32(mapa_shared(slot, cx) + 4u));
      for_each_overflow([&](uint2 c) {
        if ((c.x >> 10) == hi_digits) sub[atomicAdd(&s_info[3], 1)] = c;
      });
      __syncthreads();
      const int m = s_info[3];
      for (int i = threadIdx.x; i < m; i += kThreads) {
        const uint2 ci = sub[i];
        uint32_t rank = 0;
        for (int j2 = 0; j2 < m; ++j2) {
          const uint2 cj = sub[j2];
          rank += (cj.x > ci.x || (cj.x == ci.x && cj.y < ci.y)) ? 1u : 0u;
        }
        if (rank == need_l - 1) {
          s_thr[0] = ci.x;
          s_thr[1] = ci.y;
        }
      }
    } else if (ok) {
      // Exact ties at the threshold key: keep the need_l lowest positions.
      const uint32_t kstar = kprefix;
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
          for_each_cand([&](uint2 c) {
            if (c.x == kstar && (c.y & imask) == iprefix) atomicAdd(&sh[(c.y >> sh_) & dm], 1u);
          });
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
      if (ok && threadIdx.x == 0) {
        s_thr[0] = kstar;
        s_thr[1] = istar;
      }
    }
    if (!ok && threadIdx.x == 0) raise_error(kErrCheck);
    __syncthreads();
    // Push the threshold to every CTA of the row.
    if (threadIdx.x < static_cast<unsigned>(cs)) {
      const uint32_t a = mapa_shared(smem_u32(&s_thr[0]), threadIdx.x);
      st_shared_cluster_u32(a, s_thr[0]);
      st_shared_cluster_u32(a + 4, s_thr[1]);
    }
  }
  cluster_sync();   // #2: every CTA has the threshold

  // ---- every CTA: its winners among its candidates (its own slots, then
  //      the global overflow), then its selected count.
  const uint32_t tkey = s_thr[0];
  const uint32_t tpos = s_thr[1];
  if (has) {
    const int nmine = s_info[0];
    for (int e = threadIdx.x; e < nmine; e += kThreads) {
      const uint2 c = e < kCandSlot ? scand[e] : __ldcg(cand_row + lo + e);
      if (c.x > tkey || (c.x == tkey && c.y <= tpos)) {
        const int off = static_cast<int>(c.y) - lo;
        atomicOr(&sbits[off >> 5], 1u << (off & 31));
      }
    }
  }
  __syncthreads();
  constexpr int kWords = C / 32;                       // this chunk's bitmap words
  constexpr int kWPT = (kWords + kThreads - 1) / kThreads;
  const int nw = has ? (hi - lo + 31) / 32 : 0;
  uint32_t wv[kWPT];
  uint32_t cnt = 0;
#pragma unroll
  for (int u = 0; u < kWPT; ++u) {
    const int w = static_cast<int>(threadIdx.x) * kWPT + u;
    wv[u] = w < nw ? sbits[w] : 0u;
    cnt += __popc(wv[u]);
  }
  uint32_t pos = block_excl_scan_512(cnt, scratch);
  // Push this chunk's selected count to every CTA of the row.
  {
    const uint32_t mysel = scratch[16 + 15];   // the block's inclusive total
    if (threadIdx.x < static_cast<unsigned>(cs))
      st_shared_cluster_u32(mapa_shared(smem_u32(&s_allsel[x]), threadIdx.x), mysel);
  }
  cluster_sync();   // #3: every CTA has every chunk's count; no remote access after this
  uint32_t base = 0, total = 0;
#pragma unroll
  for (int y = 0; y < cs; ++y) {
    const uint32_t c = s_allsel[y];
    if (y < x) base += c;
    total += c;
  }
  if (x == 0 && threadIdx.x == 0 && total != static_cast<uint32_t>(k)) raise_error(kErrCheck);
  pos += base;
#pragma unroll
  for (int u = 0; u < kWPT; ++u) {
    uint32_t bits = wv[u];
    const int w = static_cast<int>(threadIdx.x) * kWPT + u;
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < static_cast<uint32_t>(k)) out_row[pos] = lo + w * 32 + b;
      ++pos;
    }
  }
}

}  // namespace

namespace {

constexpr int kQs[4] = {4, 6, 8, 16};       // float4 groups per thread the launcher chooses from
constexpr int kOneSmemBytes = 120 * 1024;   // more than half an SM's shared memory: one CTA per SM

template <int Q>
void* select_kernel_ptr() {
  return reinterpret_cast<void*>(topk_select_kernel<Q>);
}

void* select_kernel_for(int q) {
  switch (q) {
    case 4: return select_kernel_ptr<4>();
    case 6: return select_kernel_ptr<6>();
    case 8: return select_kernel_ptr<8>();
    default: return select_kernel_ptr<16>();
  }
}

// Clusters of cs CTAs that fit on the device at once, one or (as many as the
// registers allow, two) CTAs per SM; cached per device.  0 if unknown.
int max_active_clusters(int qi, int cs, bool one) {
  static std::mutex mu;
  static int cache[64][4][2][kTopkClusterCtas + 1];
  static bool filled[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!filled[dev]) {
    for (auto& a : cache[dev])
      for (auto& b : a)
        for (int& c : b) c = -1;
    filled[dev] = true;
  }
  int& slot = cache[dev][qi][one ? 1 : 0][cs];
  if (slot < 0) {
    void* kern = select_kernel_for(kQs[qi]);
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = one ? kOneSmemBytes : kSmemBytes;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = static_cast<unsigned>(cs);
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kOneSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
      n = 0;
    slot = n;
  }
  return slot;
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) {
  const int T = a.batch * a.nq;
  if (a.ld > int64_t(kTopkClusterCtas) * kThreads * 4 * kQs[3]) return cudaErrorInvalidValue;
  if (!a.hist_ready) {
    const int chunks = static_cast<int>((a.ld + kTopkChunk - 1) / kTopkChunk);
    topk_hist_kernel<<<dim3(chunks > 0 ? chunks : 1, T), kThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // The plan: the smallest chunk that covers the row, CTAs packed as the
  // registers allow (two per SM at Q = 4) -- unless one CTA per SM fits every
  // row's cluster at once and loads fewer score bytes per SM.  One CTA per
  // SM also leaves CTA 0's resolve the SM to itself, but fewer clusters of 16
  // fit at once (7 of 16 on 152 SMs, 8 of 12); with more than one wave the
  // packed plan measured faster.
  int best_q = -1, best_cs = 0;
  bool best_one = false;
  double base_bytes = 0.0;
  for (int qi = 0; qi < 4 && best_q < 0; ++qi) {
    const int64_t chunk = int64_t(kThreads) * 4 * kQs[qi];
    const int cs = static_cast<int>(std::max<int64_t>(1, (a.ld + chunk - 1) / chunk));
    if (cs > kTopkClusterCtas) continue;
    best_q = qi;
    best_cs = cs;
    cudaFuncAttributes fa{};
    const int regs = cudaFuncGetAttributes(&fa, select_kernel_for(kQs[qi])) == cudaSuccess
                         ? std::max(1, fa.numRegs) : 128;
    const int per_sm = std::max(1, std::min(2, 65536 / (regs * kThreads)));
    base_bytes = static_cast<double>(chunk) * 4.0 * per_sm;
  }
  if (best_q < 0) return cudaErrorInvalidValue;
  for (int qi = 0; qi < 4; ++qi) {
    const int64_t chunk = int64_t(kThreads) * 4 * kQs[qi];
    const int cs = static_cast<int>(std::max<int64_t>(1, (a.ld + chunk - 1) / chunk));
    if (cs > kTopkClusterCtas || static_cast<double>(chunk) * 4.0 >= base_bytes) continue;
    if (max_active_clusters(qi, cs, true) >= T) {
      best_q = qi;
      best_cs = cs;
      best_one = true;
      break;
    }
  }
  const int smem = best_one ? kOneSmemBytes : kSmemBytes;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kOneSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(best_cs, T), dim3(kThreads), smem, stream,
                         a.pdl != 0 && a.hist_ready, best_cs, a);
  };
  switch (kQs[best_q]) {
    case 4: return go(topk_select_kernel<4>);
    case 6: return go(topk_select_kernel<6>);
    case 8: return go(topk_select_kernel<8>);
    default: return go(topk_select_kernel<16>);
  }
}

// ---------------------------------------------------------------------------
// Top-k without a caller-provided workspace (dsa_topk_noalloc).
//
// For callers that cannot allocate device memory at the point where they run
// the selection, the histogram and the candidate lists live in one
// statically sized device array.  Every GPU that loads the library reserves
// it (kNoAllocScratchBytes) until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxRows = 64;                 // query rows T
constexpr long long kNoAllocMaxScores = 1ll << 21;  // T * ld_logits
constexpr size_t kNoAllocHistBytes = size_t(kNoAllocMaxRows) * kHistBins * 4;
constexpr size_t kNoAllocCandOff = (kNoAllocHistBytes + 255) & ~size_t(255);
constexpr size_t kNoAllocScratchBytes = kNoAllocCandOff + size_t(kNoAllocMaxScores) * 8;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  Looked up on
// every call (cheap): the host-side symbol is not a device address, and an
// address cached across calls would go stale if the device's context were
// reset and the module loaded again.
void* noalloc_scratch(cudaError_t* err) {
  void* ptr = nullptr;
  *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  return *err == cudaSuccess ? ptr : nullptr;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_topk_noalloc(const dsa_decode_desc* d, const float* logits,
                                       int64_t ld, int32_t* topk_idx, void* stream) {
  using namespace dsa;
  // The descriptor checks of dsa_topk, so both entry points answer alike.
  const int st = check_decode_desc(d);
  if (st != DSA_OK) return static_cast<dsa_status>(st);
  if (!logits || !topk_idx || (reinterpret_cast<uintptr_t>(logits) & 15) ||
      (reinterpret_cast<uintptr_t>(topk_idx) & 3))
    return DSA_ERR_INVALID_ARG;
  if (ld < static_cast<int64_t>(d->max_pages) * DSA_PAGE_SIZE || ld % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  const int T = d->batch * d->q_per_req;
  if (T > kNoAllocMaxRows || static_cast<long long>(T) * ld > kNoAllocMaxScores)
    return DSA_ERR_UNSUPPORTED;   // beyond the fixed scratch: use dsa_topk with a workspace
  if (ld > kTopkMaxLd) return DSA_ERR_UNSUPPORTED;
  cudaError_t e;
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch(&e));
  if (!base) return DSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The previous call's histogram is still there: clear it.
  e = cudaMemsetAsync(base, 0, kNoAllocCandOff, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  TopkLaunch a{};
  a.seqlens = d->seqlens; a.logits = logits; a.ld = ld; a.out = topk_idx;
  a.hist = reinterpret_cast<uint32_t*>(base);
  a.cand = reinterpret_cast<uint2*>(base + kNoAllocCandOff);
  a.batch = d->batch; a.nq = d->q_per_req; a.k = d->topk; a.hist_ready = 0;
  return launch_topk(a, s) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
