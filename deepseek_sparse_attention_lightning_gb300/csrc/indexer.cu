// indexer.cu -- stage 1, the lightning indexer, on tcgen05 tensor cores.
//
// Score ("MTP and sparse attention: NSA and DSA", section "Sparse attention:
// NSA and DSA"):  I[t,s] = sum_j w[t,j] * ReLU(q^I[t,j] . k^I[s]),
// 64 heads x 128 dims in FP8 E4M3 with one fp32 scale per token.  With
// positive scales, I[t,s] = ks[s] * sum_j (w[t,j] * qs[t]) * ReLU(q8[t,j] . k8[s]).
//
// Mapping: one MMA tile is 128 cached tokens (two 64-token pages) x the
// 64 * n_q index heads of one request's query tokens, K = 128 FP8 bytes:
//   D[token, head] = sum_d k8[token, d] * q8[head, d]   (tcgen05 kind::f8f6f4,
//   fp32 accumulator in TMEM).
// Each of the 128 TMEM lanes then holds one token's row of head dots, so the
// epilogue thread that owns the lane applies ReLU, the per-head weights and the
// key scale with no cross-thread reduction, writes the fp32 logit and counts it
// in a shared-memory histogram of the top 11 key bits (the first top-k pass).
//
// Warp roles (one persistent CTA per SM; 512 threads at n_q = 1, 640 at
// n_q = 2, else 384):
//   warp 0   TMA producer: one 8 KB box per page into a ring of 5-12 stages
//            (as many as shared memory holds next to the fixed buffers),
//            issued by 8 lanes for 4 tiles at a time, and the request's FP8
//            queries (double-buffered) when the request changes.  It issues
//            nothing else: a TMA instruction costs its issuing thread
//            ~100-170 cycles.
//   warps 1, 2  MMA issuers (one thread each, alternate tiles); warp 1 owns
//            TMEM;
//   warps 4-7, 8-11 (and 12-15 at n_q = 1, 12-19 at n_q = 2)  epilogue groups taking tiles in
//            turn (one thread per TMEM lane / token); each thread loads its
//            token's key scale three of its tiles ahead.  With two groups at
//            n_q = 1 the epilogue set the pace: the MMA issuers waited for
//            free accumulators and the producer for free stages a quarter of
//            the time; a third group takes most of that wait off.
// Accumulators: six TMEM buffers at n_q = 1, four at n_q = 2 (one per
// epilogue group), else two, so the MMAs of a tile do not wait for the
// epilogue of the tile a few before it.
// The requests' lengths are kept in shared memory from the tile scan; the
// producer looks up its first four tiles' page ids itself (one global load
// each, in flight while it issues the query copy) and the other warps fetch
// the rest of the range's page ids once into shared memory.  Keys are
// streamed exactly once per request; every query token of the request is
// served by the same key tile (N = 64 * n_q).
#include <atomic>

#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(indexer)

namespace dsa {
namespace {

constexpr int kTile = 128;                      // tokens per MMA tile (M)
constexpr int kStageBytes = kTile * kIndexDim;  // 16 KB of FP8 keys
constexpr int kEpiWarp0 = 4;   // epilogue groups: warps 4-7, 8-11 (, 12-15)
constexpr int kMaxBatch = 1024;
constexpr int kPageWin = 512;   // page ids cached in shared memory (256 tiles)
constexpr int kScaleAhead = 3;  // epilogue scale prefetch distance (own tiles)
constexpr int kGroup = 4;       // tiles whose copies the producer warp issues together
constexpr int kHistFlushTiles = 500;   // a group's tiles per histogram flush (< 65536 / 128)
constexpr int kSmemLimit = 232448;

template <int NQ>
struct Cfg {
  static constexpr int kN = 64 * NQ;
  static constexpr int kQBytes = kN * kIndexDim;
  // Epilogue groups (four warps each, group gi takes the tiles it = gi mod
  // kEpiGroups): three at n_q = 1 and four at n_q = 2, where the epilogue
  // sets the streaming pace with two, else two.  Every accumulator buffer
  // must be used by one group and one MMA issuer only (the tiles it = ab mod
  // kAccBufs), so kAccBufs is a multiple of both: six buffers of 64 columns
  // at n_q = 1, four of 128 at n_q = 2.  At n_q = 2 the block has 640
  // threads (at most 96 registers each), so the epilogue loads a query
  // token's 64 columns in two halves of 32.
  static constexpr int kEpiGroups = NQ == 1 ? 3 : (NQ == 2 ? 4 : 2);
  static constexpr int kThreads = 32 * (kEpiWarp0 + 4 * kEpiGroups);
  // Everything but the key ring; the ring then takes what shared memory is
  // left (up to 14 stages): the ring's bytes in flight set the bandwidth.
  static constexpr int kHistBytes = kEpiGroups * NQ * kHistBins * 2;   // 16-bit bins
  static constexpr int kFixed = 2 * kQBytes + kHistBytes + kEpiGroups * kN * 4 + kPageWin * 4 +
                                (1024 + 4) * 4 + 1024 * 4 + 64 * 4 + (2 * 14 + 4 + 2 * 6 + 1) * 8 + 16 +
                                1024;
  static constexpr int kStagesFit = (kSmemLimit - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > 14 ? 14 : kStagesFit;
  // Accumulator buffers: four when they fit in TMEM, so the MMA of a tile
  // never waits for the epilogue of the tile two before it.
  static constexpr int kAccBufs = NQ == 1 ? 6 : ((4 * kN <= 512) ? 4 : 2);
  static_assert(kAccBufs % kEpiGroups == 0 && kAccBufs % 2 == 0, "one group, one issuer per buffer");
  static constexpr int kTmemCols =
      (kAccBufs * kN <= 128) ? 128 : ((kAccBufs * kN <= 256) ? 256 : 512);
  static constexpr int kOffStages = 0;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffHist = kOffQ + 2 * kQBytes;
  static constexpr int kOffW = kOffHist + kHistBytes;
  static constexpr int kOffPages = kOffW + kEpiGroups * kN * 4;
  static constexpr int kOffPrefix = kOffPages + kPageWin * 4;
  static constexpr int kOffSeq = kOffPrefix + (kMaxBatch + 4) * 4;
  static constexpr int kOffScratch = kOffSeq + kMaxBatch * 4;
  static constexpr int kOffBar = kOffScratch + 64 * 4;
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kAccBufs + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffTmemSlot + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kOffBar % 8 == 0, "barrier alignment");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Exclusive prefix sum over the Threads threads of the block (one value each).
template <int Threads>
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  constexpr int kWarps = Threads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) scratch[32 + lane] = w;
  }
  __syncthreads();
  const int warp_off = warp ? scratch[32 + warp - 1] : 0;
  *total = scratch[32 + kWarps - 1];
  return warp_off + x - v;
}

// Request owning flattened tile g (prefix[r] <= g < prefix[r+1]).
__device__ __forceinline__ int find_request(const int* prefix, int B, int g) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Page id of page `which` (0/1) of flattened tile g, or -1 if it lies outside
// the cache.  The tile's second page, past the request's last page, repeats
// the first.
__device__ __forceinline__ int tile_page(const IndexerLaunch& p, const int* prefix, const int* seq,
                                         int r, int g, int which) {
  const int S = seq[r];
  const int npg = (S + kPage - 1) / kPage;
  int lp = 2 * (g - prefix[r]) + which;
  if (lp >= npg) lp = lp - 1;
  const int pg = p.page_table[static_cast<long long>(r) * p.max_pages + lp];
  return (pg >= 0 && pg < p.num_pages) ? pg : -1;
}

template <int NQ>
__global__ void __launch_bounds__(Cfg<NQ>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_q, const IndexerLaunch p) {
  using C = Cfg<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  int* prefix = reinterpret_cast<int*>(smem + C::kOffPrefix);
  int* seq_s = reinterpret_cast<int*>(smem + C::kOffSeq);   // every request's length
  int* scratch = reinterpret_cast<int*>(smem + C::kOffScratch);
  uint32_t* shist = reinterpret_cast<uint32_t*>(smem + C::kOffHist);
  float* wbuf = reinterpret_cast<float*>(smem + C::kOffW);
  int* pages = reinterpret_cast<int*>(smem + C::kOffPages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  const uint32_t bar0 = sbase + C::kOffBar;
#define KV_FULL(s) (bar0 + 8u * (s))
#define KV_EMPTY(s) (bar0 + 8u * (C::kStages + (s)))
#define Q_FULL(b) (bar0 + 8u * (2 * C::kStages + (b)))
#define Q_EMPTY(b) (bar0 + 8u * (2 * C::kStages + 2 + (b)))
#define ACC_FULL(b) (bar0 + 8u * (2 * C::kStages + 4 + (b)))
#define ACC_EMPTY(b) (bar0 + 8u * (2 * C::kStages + 4 + C::kAccBufs + (b)))
  const uint32_t PAGES = bar0 + 8u * (2 * C::kStages + 4 + 2 * C::kAccBufs);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.batch;
  if (threadIdx.x == 0) {   // descriptor fetches overlap the prologue's loads
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_q);
  }

  // Tiles per request (requests whose every query selects all tokens are
  // skipped when asked), then their prefix sums.
  {
    int cnt[3], sum = 0;
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      const int r = threadIdx.x * 3 + e;
      int c = 0;
      if (r < B) {
        const int S = p.seqlens[r];
        seq_s[r] = S;
        if (S > 0 && !(p.skip_short && S <= p.topk)) c = (S + kTile - 1) / kTile;
      }
      cnt[e] = c;
      sum += c;
    }
    int total;
    int run = block_excl_scan<C::kThreads>(sum, scratch, &total);
    if (threadIdx.x == 0) prefix[0] = 0;
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      const int r = threadIdx.x * 3 + e;
      run += cnt[e];
      if (r < B) prefix[r + 1] = run;
    }
  }
  for (int i = threadIdx.x; i < C::kHistBytes / 4; i += C::kThreads) shist[i] = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(KV_FULL(s), 1);
      mbar_init(KV_EMPTY(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(Q_FULL(b), 1);
      mbar_init(Q_EMPTY(b), 2);   // one commit per MMA issuer
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(ACC_FULL(b), 1);
      mbar_init(ACC_EMPTY(b), 128);
    }
    mbar_init(PAGES, 1);   // warps 1-11 stored the shared page ids
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = prefix[B];
  const int G = gridDim.x;
  const int g0 = static_cast<int>((static_cast<long long>(blockIdx.x) * total) / G);
  const int g1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * total) / G);

  grid_dep_launch();   // the top-k may be scheduled as this kernel's CTAs retire
  // Page ids of the first kPageWin / 2 tiles of the range, fetched into
  // shared memory by warps 1-11 at once; the producer warp does not wait for
  // them: it looks up its first group's pages itself and starts streaming.
  if (warp != 0) {
    const int n = min(2 * (g1 - g0), kPageWin);
    for (int i = threadIdx.x - 32; i < n; i += C::kThreads - 32) {
      const int g = g0 + (i >> 1);
      pages[i] = tile_page(p, prefix, seq_s, find_request(prefix, B, g), g, i & 1);
    }
    named_bar_sync(5, C::kThreads - 32);
    if (threadIdx.x == 32) mbar_arrive(PAGES);
  }
  auto page_of = [&](int r, int g, int which) -> int {
    const int i = 2 * (g - g0) + which;
    return i < kPageWin ? pages[i] : tile_page(p, prefix, seq_s, r, g, which);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp issues, kGroup tiles at a time: lane 2u + w copies page
    // w of tile u of the group, after lane 2u waited for the stage and armed
    // its barrier (copies from several threads keep more requests in flight
    // than one issuing thread).  The queries of a request that starts in the
    // group go first, from lane 0.
    if (g0 < g1) {
      const uint64_t pol_k = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      const int ntl = g1 - g0;
      int r = 0, cur = -1, seg = -1;   // lane 0: request and query segment
      int rl = 0;                      // this lane's request (its tiles only increase)
      int done = 0;                    // tiles whose copies were all issued
      bool ok = true;
      for (int it0 = 0; it0 < ntl; it0 += kGroup) {
        // This lane's tile and its page id first: the first group's page-table
        // reads are then in flight while lane 0 issues the query copy.
        const int it = it0 + (lane >> 1);
        const int which = lane & 1;
        const bool act = lane < 2 * kGroup && it < ntl;
        int pg = -1;
        if (act) {
          const int g = g0 + it;
          while (prefix[rl + 1] <= g) ++rl;
          if (it0 == 0) {
            // tile_page's lookup, its range check deferred to the copy below
            // so that nothing waits for the load before the query copy.
            const int npg = (seq_s[rl] + kPage - 1) / kPage;
            int lp = 2 * (g - prefix[rl]) + which;
            if (lp >= npg) lp = lp - 1;
            pg = p.page_table[static_cast<long long>(rl) * p.max_pages + lp];
          } else {
            pg = page_of(rl, g, which);
          }
        }
        if (lane == 0) {
          for (int u = 0; u < kGroup && it0 + u < ntl && ok; ++u) {
            const int g = g0 + it0 + u;
            while (prefix[r + 1] <= g) ++r;
            if (r != cur) {
              cur = r;
              ++seg;
              const int qb = seg & 1;
              if (seg >= 2 && !mbar_wait(Q_EMPTY(qb), ((seg >> 1) - 1) & 1, p.wait_cycles)) {
                ok = false;
                break;
              }
              mbar_expect_tx(Q_FULL(qb), C::kQBytes);
              tma_load_2d(sbase + C::kOffQ + qb * C::kQBytes, &tmap_q, 0, r * C::kN, Q_FULL(qb),
                          pol_q);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t st = static_cast<uint32_t>(it) % C::kStages;
        bool armed = true;
        if (act && which == 0) {
          if (it >= C::kStages)
            armed = mbar_wait(KV_EMPTY(st), ((it / C::kStages) - 1) & 1, p.wait_cycles);
          if (armed) mbar_expect_tx(KV_FULL(st), kStageBytes);
        }
        armed = __shfl_sync(0xffffffffu, armed, lane & ~1);
        if (__any_sync(0xffffffffu, act && !armed)) { ok = false; break; }
        if (act) {
          // An out-of-range page id (-1 here) is reported and read past the
          // cache end (TMA fills zeros); the epilogue masks its tokens.
          // A request's new tokens (its last n_q <= 4) lie in its last two
          // tiles, which the kernel before may still be writing (their keys,
          // not the page table).
          const int g = g0 + it;
          if (p.wait_tail && g >= prefix[rl + 1] - 2) grid_dep_wait();
          if (pg >= p.num_pages) pg = -1;
          if (pg < 0) raise_error(kErrCheck);
          const int y = pg >= 0 ? pg * kPage : p.num_pages * kPage;
          tma_load_2d(sbase + C::kOffStages + st * kStageBytes + which * (kPage * kIndexDim), &tmap_k,
                      0, y, KV_FULL(st), pol_k);
        }
        done = min(it0 + kGroup, ntl);
        // From the second group on, the pages come from shared memory.
        if (it0 == 0 && ntl > kGroup && !mbar_wait(PAGES, 0, p.wait_cycles)) {
          ok = false;
          break;
        }
      }
      if (lane == 0) {
        if (!ok) raise_error(kErrTimeout);
        // No copy may still be in flight when the CTA exits.
        const uint32_t it = static_cast<uint32_t>(done);
        const uint32_t n = it < static_cast<uint32_t>(C::kStages) ? it : C::kStages;
        for (uint32_t s = 0; s < n; ++s) {
          const uint32_t u = it - 1 - ((it - 1 - s) % C::kStages);
          mbar_wait(KV_FULL(u % C::kStages), (u / C::kStages) & 1);
        }
        if (seg >= 0) mbar_wait(Q_FULL(seg & 1), (seg >> 1) & 1);
        if (seg >= 1) mbar_wait(Q_FULL((seg - 1) & 1), ((seg - 1) >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads: warp 1 takes the even tiles (accumulator 0),
    // warp 2 the odd ones (accumulator 1); one thread alone could not issue
    // a tile's MMAs and commits as fast as HBM delivers the tiles.  Both walk
    // every tile to keep the request (query buffer) count in step.
    const uint32_t mi = static_cast<uint32_t>(warp - 1);
    if (lane == 0 && g0 < g1) {
      constexpr uint32_t idesc = make_idesc(0, 0, 0, 0, C::kN, 128);
      int r = 0, cur = -1, seg = -1;
      bool q_ready = false, ok = true;
      int last = -1;
      for (int g = g0; g < g1; ++g) {
        while (prefix[r + 1] <= g) ++r;
        if (r != cur) {
          if (seg >= 0) tc_commit(Q_EMPTY(seg & 1));
          cur = r;
          ++seg;
          q_ready = false;
        }
        const uint32_t it = static_cast<uint32_t>(g - g0);
        if ((it & 1) != mi) continue;
        if (!q_ready) {
          if (!mbar_wait(Q_FULL(seg & 1), (seg >> 1) & 1, p.wait_cycles)) { ok = false; break; }
          q_ready = true;
        }
        const uint32_t st = it % C::kStages;
        if (!mbar_wait(KV_FULL(st), (it / C::kStages) & 1, p.wait_cycles)) { ok = false; break; }
        const uint32_t ab = it % C::kAccBufs;
        if (it >= C::kAccBufs &&
            !mbar_wait(ACC_EMPTY(ab), ((it / C::kAccBufs) - 1) & 1, p.wait_cycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sbase + C::kOffStages + st * kStageBytes;
        const uint32_t b0 = sbase + C::kOffQ + (seg & 1) * C::kQBytes;
        const uint32_t d = tmem_base + ab * C::kN;
#pragma unroll
        for (int kk = 0; kk < kIndexDim / 32; ++kk) {
          mma_f8_ss(d, smem_desc_sw128(a0 + kk * 32, 16, 1024),
                    smem_desc_sw128(b0 + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(KV_EMPTY(st));
        tc_commit(ACC_FULL(ab));
        last = static_cast<int>(it);
      }
      if (seg >= 0) tc_commit(Q_EMPTY(seg & 1));
      if (!ok) raise_error(kErrTimeout);
      if (last >= 0) mbar_wait(ACC_FULL(last % C::kAccBufs), (last / C::kAccBufs) & 1);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Group gi handles the tiles it = gi, gi + 2, ... (accumulator gi), with
    // its own histogram and weight buffer, so two tiles are in flight.
    const int gi = (warp - kEpiWarp0) / 4;
    const int q4 = warp & 3;               // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;        // token within the tile
    const int tid = (warp - kEpiWarp0 - 4 * gi) * 32 + lane;
    const uint32_t bar_id = 1 + gi;
    // Histogram bins are 16-bit halves of 32-bit words (bin b: word b / 2),
    // flushed to the global histogram at a request change and every
    // kHistFlushTiles tiles, so no bin can overflow.
    uint32_t* ghist = shist + gi * NQ * (kHistBins / 2);
    int seg_tiles = 0;
    float* gw = wbuf + gi * C::kN;
    const float ninf = __int_as_float(0xff800000);
    // Key scale of this thread's token in tile g (0 if the page is invalid).
    int rs = 0;
    auto scale_of = [&](int g) -> float {
      if (g >= g1) return 0.f;
      while (prefix[rs + 1] <= g) ++rs;
      if (p.wait_tail && g >= prefix[rs + 1] - 2) grid_dep_wait();   // new tokens' scales
      const int pg = page_of(rs, g, row >> 6);
      return pg >= 0 ? __ldg(p.k_scale + static_cast<long long>(pg) * kPage + (row & (kPage - 1)))
                     : 0.f;
    };
    float sk0 = scale_of(g0 + gi), sk1 = scale_of(g0 + gi + C::kEpiGroups),
          sk2 = scale_of(g0 + gi + 2 * C::kEpiGroups);
    static_assert(kScaleAhead == 3, "three scale registers");
    int r = 0, cur = -1, S = 0;
    bool ok = true;
    auto flush_hist = [&](int req) {
      // The histogram may be cleared by the kernel before (fused path): the
      // first global atomic waits for it; everything earlier does not.
      grid_dep_wait();
      named_bar_sync(bar_id, 128);
      for (int i = 0; i < NQ; ++i) {
        uint32_t* gh = p.hist + static_cast<long long>(req * NQ + i) * kHistBins;
        for (int w = tid; w < kHistBins / 2; w += 128) {
          const uint32_t v = ghist[i * (kHistBins / 2) + w];
          if (v) {
            if (v & 0xFFFFu) atomicAdd(gh + 2 * w, v & 0xFFFFu);
            if (v >> 16) atomicAdd(gh + 2 * w + 1, v >> 16);
            ghist[i * (kHistBins / 2) + w] = 0u;
          }
        }
      }
      named_bar_sync(bar_id, 128);
      seg_tiles = 0;
    };
    for (int g = g0 + gi; g < g1; g += C::kEpiGroups) {
      const uint32_t it = static_cast<uint32_t>(g - g0);
      while (prefix[r + 1] <= g) ++r;
      if (r != cur) {
        if (cur >= 0 && p.hist) flush_hist(cur);
        seg_tiles = 0;
        named_bar_sync(bar_id, 128);
        cur = r;
        S = seq_s[r];
        for (int e = tid; e < C::kN; e += 128) {
          const int t = r * NQ + e / kIndexHeads;
          gw[e] = p.w[static_cast<long long>(t) * kIndexHeads + (e % kIndexHeads)] * p.q_scale[t];
        }
        named_bar_sync(bar_id, 128);
      }
      const int s = (g - prefix[r]) * kTile + row;
      const float sk = sk0;
      const bool tok_ok = s < S && page_of(r, g, row >> 6) >= 0;
      sk0 = sk1;
      sk1 = sk2;
      sk2 = scale_of(g + kScaleAhead * C::kEpiGroups);
      const uint32_t ab = it % C::kAccBufs;
      // A wait that ran out stops this warp's work on every later tile, but
      // the loop goes on (through the group's named barriers, which every
      // thread must pass equally often); the decision is warp-wide because
      // the TMEM loads are warp-collective.
      if (!ok || !mbar_wait(ACC_FULL(ab), (it / C::kAccBufs) & 1, p.wait_cycles)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + ab * C::kN;
#pragma unroll 1
        for (int i = 0; i < NQ; ++i) {
          const float4* w4 = reinterpret_cast<const float4*>(gw + i * kIndexHeads);
          float s0 = 0.f, s1 = 0.f;
          if constexpr (NQ == 2) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t acc[32];
              tmem_ld32(tl + i * 64 + hf * 32, acc);
              if (i == NQ - 1 && hf == 1) {
                tc_fence_before();
                mbar_arrive(ACC_EMPTY(ab));
              }
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const float4 ww = w4[8 * hf + jj];
                s0 = fmaf(ww.x, fmaxf(__uint_as_float(acc[4 * jj + 0]), 0.f), s0);
                s1 = fmaf(ww.y, fmaxf(__uint_as_float(acc[4 * jj + 1]), 0.f), s1);
                s0 = fmaf(ww.z, fmaxf(__uint_as_float(acc[4 * jj + 2]), 0.f), s0);
                s1 = fmaf(ww.w, fmaxf(__uint_as_float(acc[4 * jj + 3]), 0.f), s1);
              }
            }
          } else {
            uint32_t acc[64];
            tmem_ld64(tl + i * 64, acc);
            if (i == NQ - 1) {
              tc_fence_before();
              mbar_arrive(ACC_EMPTY(ab));
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float4 ww = w4[jj];
              s0 = fmaf(ww.x, fmaxf(__uint_as_float(acc[4 * jj + 0]), 0.f), s0);
              s1 = fmaf(ww.y, fmaxf(__uint_as_float(acc[4 * jj + 1]), 0.f), s1);
              s0 = fmaf(ww.z, fmaxf(__uint_as_float(acc[4 * jj + 2]), 0.f), s0);
              s1 = fmaf(ww.w, fmaxf(__uint_as_float(acc[4 * jj + 3]), 0.f), s1);
            }
          }
          if (s < p.ld) {
            const int vis = S - (NQ - 1 - i);
            const bool live = tok_ok && s < vis;
            const float v = live ? (s0 + s1) * sk : ninf;
            p.logits[static_cast<long long>(r * NQ + i) * p.ld + s] = v;
            if (p.hist && live) {
              const uint32_t bin = float_key(v) >> kHistShift;
              atomicAdd(&ghist[i * (kHistBins / 2) + (bin >> 1)], 1u << (16 * (bin & 1)));
            }
          }
        }
      }
      if (p.hist && ++seg_tiles == kHistFlushTiles) flush_hist(cur);
    }
    if (!ok) raise_error(kErrTimeout);
    if (cur >= 0 && p.hist) flush_hist(cur);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  // This grid completes only after the kernel before it (the stages after
  // the top-k rely on that, even when no tile here waited for it).
  if (p.pdl && threadIdx.x == 0) grid_dep_wait();
#undef KV_FULL
#undef KV_EMPTY
#undef Q_FULL
#undef Q_EMPTY
#undef ACC_FULL
#undef ACC_EMPTY
}

std::atomic<long long> g_wait_cycles{0};

template <int NQ>
cudaError_t launch_nq(const IndexerLaunch& a_in, cudaStream_t stream) {
  using C = Cfg<NQ>;
  IndexerLaunch a = a_in;
  const long long wc = g_wait_cycles.load(std::memory_order_relaxed);
  a.wait_cycles = wc > 0 ? wc : kWaitCycles;
  CUtensorMap tk, tq;
  const uint64_t rows = static_cast<uint64_t>(a.num_pages) * kPage;
  const uint64_t qrows = static_cast<uint64_t>(a.batch) * NQ * kIndexHeads;
  if (!encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_fp8, kIndexDim, rows, kIndexDim,
                      kIndexDim, kPage, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_fp8, kIndexDim, qrows, kIndexDim,
                      kIndexDim, C::kN, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = device_sm_count();
  return launch_kernel(indexer_kernel<NQ>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream,
                       a.pdl != 0, 1, tk, tq, a);
}

}  // namespace

void set_indexer_wait_cycles(long long cycles) {
  g_wait_cycles.store(cycles > 0 ? cycles : 0, std::memory_order_relaxed);
}

cudaError_t launch_indexer(const IndexerLaunch& a, cudaStream_t stream) {
  switch (a.nq) {
    case 1: return launch_nq<1>(a, stream);
    case 2: return launch_nq<2>(a, stream);
    case 3: return launch_nq<3>(a, stream);
    case 4: return launch_nq<4>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
