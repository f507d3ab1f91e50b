// sparse_mla.cu -- stage 3, absorbed-form MLA over only the selected latent
// rows, as split-KV online-softmax partials ("Deepseek Details", section
// "DSA", stage 2: Mid_O[batch, head, block, dim] and
// Mid_O_LogExpSum[batch, head, block]; the latent row is kv_lora_rank 512 +
// rope 64 = 576 dims and V is its first 512 dims: "[SGLang] NSA", section
// "forward_decode").
//
// One CTA = (query row t, split b, value half v).  The CTA attends the
// selected positions of its split in tiles of 64 keys with all H (<= 128)
// heads as the MMA M dimension, and owns output dims [256 v, 256 v + 256).
//
// Why halves: the fp32 output of 128 heads x 512 dims is 256 KB, all of a
// SM's tensor memory, so one CTA keeps half of it (256 TMEM columns) and the
// two CTAs of a (t, b) both compute S = Q K^T.  Each gathers whole rows
// itself (the second fetch of a row mostly hits L2); no data moves between
// CTAs.
//
// Tensor memory (512 columns):
//   [  0,256)  O   fp32 accumulator, this CTA's 256 value dims
//   [256,320)  S   fp32 scores of the current 64-key tile
//   [320,352)  P   bf16 probabilities (2 per column), the A operand of P V
//   [352,512)  Q   q dims [0, 320) as bf16 pairs, the A operand of Q K^T
// Shared memory: q dims [320, 576) (64 KB, 128B-swizzled) and two stages of
// 64 gathered latent rows (9 atoms of 64 dims, 72 KB each).  Before the
// second stage holds keys it holds q dims [0, 256), brought by TMA for the
// softmax threads to move into TMEM (q dims [256, 320) they load
// themselves): the SM's load/store path delivers only ~20 GB/s of scattered
// 16-byte loads, the copy engine several times that.
//
// A stage is two parts with their own full / free barriers: the K part (the
// other value half's four atoms and the rope atom, read only by Q K^T) and
// the V part (this CTA's four value atoms, read by Q K^T and P V).  The K part
// of a stage is free again as soon as Q K^T of its tile is done, so the
// gathers of the tile two ahead start about a softmax and a P V earlier than
// if the whole stage waited for P V; Q K^T takes the K part first.
//
// Per tile: S = Q K^T is 20 TMEM-A MMAs (dims 0..319) + 16 smem-A MMAs (dims
// 320..575), M = 128, N = 64, K = 16 (kind::f16, bf16 in, fp32 out).  The
// softmax threads (two per head = per TMEM lane, each with 32 of the tile's
// 64 keys) read S, apply the scale in the exp2 domain, keep a running
// maximum that is raised lazily (the accumulator is rescaled only when a
// tile's maximum exceeds it by 2^8), write P to TMEM, and P V (4 MMAs,
// N = 256, V read MN-major from the CTA's value atoms) accumulates into O.
// The MMA thread issues P V of a tile as soon as its P is written, also
// between the MMAs of the next tile's Q K^T, because that P V frees the
// V part the gather two tiles ahead waits for.
//
// Warp roles (512 threads): warps 0, 2, 3 and 8-11 resolve every selected
// position to its cache row (logical index -> page table -> row, fused here)
// and gather the rows with TMA tile::gather4 copies (4 rows x 64 dims each,
// written in the 128B-swizzled stage layout by the copy engine): 80 threads
// spread over the seven warps issue one copy of each part per tile (64 of
// them a V copy), because the copy engine takes a warp's TMA instructions one
// lane at a time but the warps' in parallel.  Warp 1 issues the MMAs and owns TMEM; warps 4-7 and 12-15 run
// the softmax and the epilogue (Mid_O written by 128B-swizzled tensor stores
// of 32 heads x 32 dims).
//
// FP8 latent rows (kFp8): per tile 64 copies (the codes of each 4 rows as
// two plain 256-byte boxes, their rope dims 128B-swizzled straight into atom
// 8, their scales), issued by warps 0, 2, 3 into one full barrier; warps 8-11
// dequantise the codes in place into bf16 atoms 0-7 and signal twice, so
// that Q K^T on dims 0..255 starts after the first half; the stage is freed
// as a whole after P V.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(mla)

namespace dsa {
namespace {

constexpr int kBN = 64;                                  // keys per tile
constexpr int kAtoms = kLatentDim / 64;                  // 9 atoms of 64 dims
constexpr int kAtomBytes = kBN * 128;                    // 8 KB
constexpr int kStageBytes = kAtoms * kAtomBytes;         // 72 KB
constexpr int kQTmemDims = 320;
constexpr int kQSmemAtoms = (kLatentDim - kQTmemDims) / 64;  // 4
constexpr int kQAtomBytes = 128 * 128;                   // 128 heads x 64 dims bf16
constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kQSmemAtoms * kQAtomBytes;
constexpr int kMaxPos = 2048;                            // positions of one split (<= k)
constexpr int kMaxRank = 512;                            // rows ranked by length (else index order)
constexpr int kOffRows = kOffStage + 2 * kStageBytes;    // cache row of every position
constexpr int kOffMask = kOffRows + kMaxPos * 4;         // validity bits, 32 per word
constexpr int kOffXchg = kOffMask + (kMaxPos / 32) * 4;    // softmax groups' exchange, 2 KB
constexpr int kOffSc = kOffXchg + 2 * 2 * 128 * 4;         // FP8 rows' tile scales, 2 stages
constexpr int kScStageBytes = (kBN / 4) * 128;             // 4 rows x 16 B per 128-byte slot
constexpr int kOffBar = kOffSc + 2 * kScStageBytes;
constexpr int kNumBars = 20;
constexpr int kQStageAtoms = 4;                            // q dims [0, 256) via stage 1
constexpr int kOffSlot = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffSlot + 16 + 1024;
constexpr int kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr int kTmemCols = 512;
constexpr int kThreads = 512;
constexpr int kSoftThreads = 256;                          // warps 4-7 and 12-15
constexpr int kLoaderWarps = 7;                            // warps 0, 2, 3, 8-11
constexpr int kVCopies = 4 * (kBN / 4);                    // V part: 4 atoms x 16 row groups
constexpr int kKCopies = 5 * (kBN / 4);                    // K part: 4 atoms + rope, 16 groups
static_assert(kVCopies <= kKCopies && kKCopies <= 32 * kLoaderWarps, "issuers");
constexpr int kResolveBatch = 4;                           // position groups in flight per loader
constexpr int kOBoxBytes = 32 * 128;                       // Mid_O box: 32 heads x 32 fp32
constexpr int kOChunkBytes = 4 * kOBoxBytes;               // the 4 warps' boxes of a chunk
static_assert(8 * kOChunkBytes <= 2 * kStageBytes, "Mid_O staging fits in the key stages");
constexpr float kRescaleLog2 = 8.0f;
// FP8 latent rows: 512 E4M3 codes (four 128-dim tiles), the 4 tiles' fp32
// scales, the 64 rope dims in bf16 -- 656 bytes.
constexpr int kF8RowBytes = 656;
constexpr int kF8Copies = (kBN / 4) * 4;                   // 2 code halves + rope + scales per 4 rows
constexpr int kRawHalfBytes = kBN * 256;                   // codes 0..255 / 256..511 of 64 rows
constexpr int kRawOff = 4 * kAtomBytes;                    // codes land in stage bytes 32..64 KB
constexpr int kConvThreads = 128;                          // warps 8-11 dequantise
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Dequantises code tile a's 16-code chunk c of key row j (scale sc) into the
// bf16 atoms of the stage, in the 128B-swizzled layout the MMAs read: dims
// 128 a + 16 c .. + 15 are atom 2a + c / 4, 16-byte chunks 2 (c % 4) and
// 2 (c % 4) + 1 of row j.
__device__ __forceinline__ void dequant_chunk(uint8_t* stage, int a, int j, int c, uint4 raw,
                                              float sc) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw h01 =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(__half2(h01));
    const float2 f23 = __half22float2(__half2(h23));
    o[2 * q] = pack_bf16x2(f01.x * sc, f01.y * sc);
    o[2 * q + 1] = pack_bf16x2(f23.x * sc, f23.y * sc);
  }
  uint8_t* atom = stage + (2 * a + (c >> 2)) * kAtomBytes + j * 128;
  const int cb = 2 * (c & 3);
  *reinterpret_cast<uint4*>(atom + ((cb ^ (j & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(atom + (((cb + 1) ^ (j & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
}

// kFp8: the latent cache holds FP8 rows (kF8RowBytes); tmap_kv then maps its
// bytes with plain 256-byte boxes (codes), tmap_rope with 128B-swizzled
// 128-byte boxes (the rope dims) and tmap_sc with 16-byte boxes (the
// scales).  Otherwise tmap_kv maps the bf16 cache and the others are unused.
template <bool kFp8, bool kRank>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_kv,
                      const __grid_constant__ CUtensorMap tmap_o,
                      const __grid_constant__ CUtensorMap tmap_sc,
                      const __grid_constant__ CUtensorMap tmap_rope, const MlaLaunch p) {
  extern __shared__ uint8_t smem_raw[];
  const int split = blockIdx.x >> 1, half = blockIdx.x & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.heads, S = p.num_splits, k = p.k;
  // The query row.  With kRank (a grid of more CTAs than the GPU has SMs),
  // blockIdx.y is the row's rank in the order of selected counts
  // min(vis, k), longest first (equal counts: lower row first): the
  // scheduler hands out CTAs in index order, so rows of different lengths
  // are taken longest first and the SMs end close together.  (Up to
  // kMaxRank rows; the counts go through the row-index area, unused until
  // the loaders fill it.)
  int t = blockIdx.y;
  if constexpr (kRank) {
    __shared__ int s_row;
    const int T = p.batch * p.nq;
    if (T > 1 && T <= kMaxRank) {
      int* cnt = reinterpret_cast<int*>(align1024(smem_raw) + kOffRows);
      for (int i = threadIdx.x; i < T; i += kThreads) {
        const int v = p.seqlens[i / p.nq] - (p.nq - 1 - i % p.nq);
        cnt[i] = v <= 0 ? 0 : (v < k ? v : k);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < T; i += kThreads) {
        const int ci = cnt[i];
        int rank = 0;
        for (int j = 0; j < T; ++j) {
          const int cj = cnt[j];
          rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
        }
        if (rank == static_cast<int>(blockIdx.y)) s_row = i;
      }
      __syncthreads();
      t = s_row;
    }
  }
  const int r = t / p.nq, qi = t % p.nq;
  const int vis = p.seqlens[r] - (p.nq - 1 - qi);
  const int n = vis <= 0 ? 0 : (vis < k ? vis : k);
  const int per = (k + S - 1) / S;
  const int chunk = kBN * ((per + kBN - 1) / kBN);
  const int start = split * chunk;
  const int end = min(start + chunk, n);
  const int ntiles = end > start ? (end - start + kBN - 1) / kBN : 0;
  const float ninf = __int_as_float(0xff800000);

  float* out_base = p.mid_o + (static_cast<long long>(t) * H * S + split) * kVDim + half * 256;
  if (ntiles == 0) {
    // Empty block: Mid_O = 0, Mid_LSE = -inf.
    for (int e = threadIdx.x; e < H * 64; e += kThreads) {
      const int h = e >> 6, c = e & 63;
      reinterpret_cast<float4*>(out_base + static_cast<long long>(h) * S * kVDim)[c] =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (half == 0)
      for (int h = threadIdx.x; h < H; h += kThreads)
        p.mid_lse[(static_cast<long long>(t) * H + h) * S + split] = ninf;
    if (p.pdl && p.sel_ready && threadIdx.x == 0) grid_dep_wait();
    return;
  }

  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  int* rows_s = reinterpret_cast<int*>(smem + kOffRows);
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(smem + kOffMask);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  const uint32_t bar0 = sbase + kOffBar;
  const uint32_t Q_FULL = bar0, Q_TMEM = bar0 + 8, S_FULL = bar0 + 16, S_FREE = bar0 + 24,
                 P_FULL = bar0 + 32, PV_DONE = bar0 + 40, Q_STAGE = bar0 + 48,
                 MMA_DRAIN = bar0 + 56;
// K_FULL(s) / V_FULL(s): the K / V part of stage s landed (FP8: V_FULL is the
// whole stage's copies).  K_EMPTY(s): Q K^T of the stage's tile is done (its K
// part may be overwritten).  V_EMPTY(s): P V of the stage's tile is done (the
// whole stage may be overwritten).  KV_CONV_A(s) / KV_CONV(s) (FP8): bf16
// atoms 0-3 / 0-7 of stage s are dequantised.
#define K_FULL(s) (bar0 + 64u + 8u * (s))
#define V_FULL(s) (bar0 + 80u + 8u * (s))
#define K_EMPTY(s) (bar0 + 96u + 8u * (s))
#define V_EMPTY(s) (bar0 + 112u + 8u * (s))
#define KV_CONV_A(s) (bar0 + 128u + 8u * (s))
#define KV_CONV(s) (bar0 + 144u + 8u * (s))

  if (threadIdx.x == 0) {
    mbar_init(Q_FULL, 1);
    mbar_init(Q_TMEM, kSoftThreads);
    mbar_init(S_FULL, 1);
    mbar_init(S_FREE, kSoftThreads);
    mbar_init(P_FULL, kSoftThreads);
    mbar_init(PV_DONE, 1);
    mbar_init(Q_STAGE, 1);
    mbar_init(MMA_DRAIN, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(K_FULL(s), kKCopies);             // one expect-tx arrive per copy
      mbar_init(V_FULL(s), kFp8 ? kF8Copies : kVCopies);
      mbar_init(K_EMPTY(s), 1);
      mbar_init(V_EMPTY(s), 1);
      mbar_init(KV_CONV_A(s), kConvThreads);
      mbar_init(KV_CONV(s), kConvThreads);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_launch();

  if (warp == 0 || warp == 2 || warp == 3 || (warp >= 8 && warp < 12)) {
    // ------------------------------------------------------------ loaders
    const int lw = warp == 0 ? 0 : (warp < 4 ? warp - 1 : warp - 5);   // loader warp 0..6
    const int ltid = lw * 32 + lane;
    const int* ptab = p.page_table + static_cast<long long>(r) * p.max_pages;
    const int* idx_row = p.topk_idx + static_cast<long long>(t) * k;
    // Queries, page table and cache are inputs of the layer; only the
    // selected positions come from the kernel before (the top-k when this
    // grid is launched as its dependent), so the query copies start first.
    if (ltid == 0) {
      prefetch_tmap(&tmap_q);
      prefetch_tmap(&tmap_kv);
      prefetch_tmap(&tmap_o);
      if (kFp8) {
        prefetch_tmap(&tmap_sc);
        prefetch_tmap(&tmap_rope);
      }
      mbar_expect_tx(Q_FULL, kQSmemAtoms * kQAtomBytes);
      mbar_expect_tx(Q_STAGE, kQStageAtoms * kQAtomBytes);
      const uint64_t pol_q = policy_evict_last();   // the other value half reads the same query
      for (int a = 0; a < kQSmemAtoms; ++a)
        tma_load_2d(sbase + kOffQ + a * kQAtomBytes, &tmap_q, kQTmemDims + 64 * a, t * H, Q_FULL,
                    pol_q);
      for (int a = 0; a < kQStageAtoms; ++a)
        tma_load_2d(sbase + kOffStage + kStageBytes + a * kQAtomBytes, &tmap_q, 64 * a, t * H,
                    Q_STAGE, pol_q);
    }
    int safe_row = 0;
    {
      const int pg0 = ptab[0];
      if (pg0 >= 0 && pg0 < p.num_pages) safe_row = pg0 * kPage;
    }
    if (!p.sel_ready) grid_dep_wait();
    // Resolve every position of the split first (logical index -> page table
    // -> cache row).  Groups of 32 positions go round-robin to the loader
    // warps, 4 groups per batch so the loads overlap.
    const int npos = ntiles * kBN;
    for (int g0 = lw; 32 * g0 < npos; g0 += kLoaderWarps * kResolveBatch) {
      int idx[kResolveBatch];
#pragma unroll
      for (int u = 0; u < kResolveBatch; ++u) {
        const int i = 32 * (g0 + kLoaderWarps * u);
        const int pos = start + i + lane;
        idx[u] = (i < npos && pos < end) ? __ldg(idx_row + pos) : -1;
      }
      int pg[kResolveBatch];
#pragma unroll
      for (int u = 0; u < kResolveBatch; ++u) pg[u] = (idx[u] >= 0 && idx[u] < vis) ? __ldg(ptab + (idx[u] >> 6)) : -1;
#pragma unroll
      for (int u = 0; u < kResolveBatch; ++u) {
        const int i = 32 * (g0 + kLoaderWarps * u);
        if (i >= npos) break;
        const int pos = start + i + lane;
        if (pos < end && idx[u] >= vis) raise_error(kErrCheck);
        bool valid = idx[u] >= 0 && idx[u] < vis;
        if (valid && (pg[u] < 0 || pg[u] >= p.num_pages)) {
          raise_error(kErrCheck);
          valid = false;
        }
        rows_s[i + lane] = valid ? pg[u] * kPage + (idx[u] & (kPage - 1)) : safe_row;
        const uint32_t m = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) mask_s[i >> 5] = m;
      }
    }
    named_bar_sync(1, kLoaderWarps * 32);   // rows_s / mask_s complete
    // Every row is fetched by the two CTAs of its (t, b) at about the same
    // time: the first fetch keeps it in L2 for the second.
    const uint64_t pol_kv = policy_evict_last();
    // Tiles this thread issued copies for, and of which parts (bit 0: K,
    // bit 1: V or the FP8 stage).
    int issued = 0, part = 0;
    if constexpr (kFp8) {
      const bool conv = lw >= 3;                      // warps 8-11 dequantise
      const int g8 = lane * 3 + lw;
      if (!conv && g8 < kF8Copies) {
        // Warps 0, 2, 3 gather, one copy per thread and tile: per row group
        // g, codes 0..255 and 256..511 as plain 256-byte rows into the raw
        // halves at stage bytes 32 KB and 48 KB, the rope dims 128B-swizzled
        // into atom 8, the scales into the scale area.
        part = 2;
        for (int it = 0; it < ntiles; ++it) {
          const int st = it & 1;
          if (it >= 2 && !mbar_wait(V_EMPTY(st), ((it >> 1) - 1) & 1)) {
            raise_error(kErrTimeout);
            break;
          }
          if (it == 1 && !mbar_wait(Q_TMEM, 0)) {   // stage 1 held the q staging
            raise_error(kErrTimeout);
            break;
          }
          const uint32_t dst = sbase + kOffStage + st * kStageBytes;
          const int* rows = rows_s + it * kBN;
          if (g8 < 32) {
            const int g = g8 >> 1, h = g8 & 1;
            const int* r4 = rows + 4 * g;
            mbar_expect_tx(V_FULL(st), 4 * 256);
            tma_gather4(dst + kRawOff + h * kRawHalfBytes + g * 1024, &tmap_kv, 256 * h, r4[0],
                        r4[1], r4[2], r4[3], V_FULL(st), pol_kv);
          } else if (g8 < 48) {
            const int* r4 = rows + 4 * (g8 - 32);
            mbar_expect_tx(V_FULL(st), 4 * 128);
            tma_gather4(dst + 8 * kAtomBytes + (g8 - 32) * 512, &tmap_rope, 528, r4[0], r4[1],
                        r4[2], r4[3], V_FULL(st), pol_kv);
          } else {
            const int* r4 = rows + 4 * (g8 - 48);
            // (a tensor copy's shared-memory destination is 128-byte aligned)
            mbar_expect_tx(V_FULL(st), 4 * 16);
            tma_gather4(sbase + kOffSc + st * kScStageBytes + (g8 - 48) * 128, &tmap_sc, 512, r4[0],
                        r4[1], r4[2], r4[3], V_FULL(st), pol_kv);
          }
          issued = it + 1;
        }
      } else if (conv) {
        // Warps 8-11 dequantise each landed stage in place: code tiles 0, 1
        // (raw half 0) become bf16 atoms 0-3 (0-32 KB); tiles 2, 3 are read
        // into registers first, because their bf16 atoms 4-7 cover the codes
        // themselves.  The eight lanes of a quarter warp take rows j0, j0 + 1
        // (j0 even) and the chunks c of one row in 0..3, of the other in 4..7,
        // so that each quarter warp's 16-byte reads and writes fall on eight
        // distinct bank groups.
        const int ctid = (lw - 3) * 32 + lane;
        const int l8 = ctid & 7, qw = ctid >> 3;
        for (int it = 0; it < ntiles; ++it) {
          const int st = it & 1;
          if (!mbar_wait(V_FULL(st), (it >> 1) & 1)) {
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* stg = smem + kOffStage + st * kStageBytes;
          const float* scs = reinterpret_cast<const float*>(smem + kOffSc + st * kScStageBytes);
          uint4 keep[8];
          float ksc[8];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int a = u >> 2, v = u & 1, rp = (u >> 1) & 1;
            const int j = 2 * (qw + 16 * rp) + (l8 >> 2);
            const int c = (l8 & 3) + 4 * ((l8 >> 2) ^ v);
            const uint4 raw = *reinterpret_cast<const uint4*>(
                stg + kRawOff + (a >> 1) * kRawHalfBytes + j * 256 + (a & 1) * 128 + c * 16);
            const float sc = scs[(j >> 2) * 32 + (j & 3) * 4 + a];
            if (u < 8) {
              dequant_chunk(stg, a, j, c, raw, sc);
            } else {
              keep[u - 8] = raw;
              ksc[u - 8] = sc;
            }
          }
          // Atoms 0-3 are ready: the Q K^T MMAs on dims 0..255 may start.
          fence_proxy_async_smem();
          mbar_arrive(KV_CONV_A(st));
          named_bar_sync(4, kConvThreads);
#pragma unroll
          for (int u = 8; u < 16; ++u) {
            const int v = u & 1, rp = (u >> 1) & 1;
            dequant_chunk(stg, u >> 2, 2 * (qw + 16 * rp) + (l8 >> 2), (l8 & 3) + 4 * ((l8 >> 2) ^ v),
                          keep[u - 8], ksc[u - 8]);
          }
          fence_proxy_async_smem();   // generic-proxy writes -> the MMAs' reads
          mbar_arrive(KV_CONV(st));
        }
      }
    } else {
      // Every thread c = 7 lane + warp issues up to one copy of each part per
      // tile (c < 80: of the K part, c < 64: of the V part), in the same
      // order in every lane -- K part free, its copy, V part free, its copy --
      // so that the warps stay converged (the copy engine serves a warp's
      // lanes one after another).  Copy c of a part brings rows 4g..4g+3 of
      // the tile, dims [64a, 64a+64), to atom a at byte 512 g (the copy
      // engine applies the 128B swizzle).  K: the other half's atoms
      // a = 4 (1 - half) + c / 16, g = c % 16 (c < 64), else the rope atom 8
      // with g = c - 64.  V: a = 4 half + c / 16, g = c % 16.
      const int c = lane * kLoaderWarps + lw;
      if (c < kKCopies) {
        part = c < kVCopies ? 3 : 1;
        const int ka = c < 64 ? 4 * (1 - half) + (c >> 4) : 8;
        const int kg = c < 64 ? (c & 15) : c - 64;
        const int va = 4 * half + (c >> 4), vg = c & 15;
        for (int it = 0; it < ntiles; ++it) {
          const uint32_t st = it & 1;
          const uint32_t dst = sbase + kOffStage + st * kStageBytes;
          if (it >= 2 && !mbar_wait(K_EMPTY(st), ((it >> 1) - 1) & 1)) {
            raise_error(kErrTimeout);
            break;
          }
          // Stage 1 holds the q dims [0, 256) until the softmax threads
          // moved them into TMEM.
          if (it == 1 && !mbar_wait(Q_TMEM, 0)) {
            raise_error(kErrTimeout);
            break;
          }
          {
            const int* r4 = rows_s + it * kBN + 4 * kg;
            mbar_expect_tx(K_FULL(st), 4 * 128);
            tma_gather4(dst + ka * kAtomBytes + kg * 512, &tmap_kv, 64 * ka, r4[0], r4[1], r4[2],
                        r4[3], K_FULL(st), pol_kv);
          }
          if (it >= 2 && !mbar_wait(V_EMPTY(st), ((it >> 1) - 1) & 1)) {
            raise_error(kErrTimeout);
            issued = it + 1;   // this tile's K copy is in flight
            break;
          }
          if (c < kVCopies) {
            const int* r4 = rows_s + it * kBN + 4 * vg;
            mbar_expect_tx(V_FULL(st), 4 * 128);
            tma_gather4(dst + va * kAtomBytes + vg * 512, &tmap_kv, 64 * va, r4[0], r4[1], r4[2],
                        r4[3], V_FULL(st), pol_kv);
          }
          issued = it + 1;
        }
      }
    }
    // No copy may still be in flight when the CTA exits: every issuing thread
    // waits (with the default bound) for the phases of its last two tiles.
    // They completed already unless a wait ran out somewhere, and then each
    // either completes or its bound passes long after the copies landed.
    for (int u = issued - 1; u >= 0 && u >= issued - 2; --u) {
      if (part & 1) mbar_wait(K_FULL(u & 1), (u >> 1) & 1);
      if (part & 2) mbar_wait(V_FULL(u & 1), (u >> 1) & 1);
    }
    if (ltid == 0) {
      mbar_wait(Q_FULL, 0);
      mbar_wait(Q_STAGE, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc(1, 1, 0, 0, kBN, 128);
      constexpr uint32_t idesc_pv = make_idesc(1, 1, 0, 1, 256, 128);
      const uint32_t tS = tmem + kColS, tO = tmem + kColO, tP = tmem + kColP, tQ = tmem + kColQ;
      const uint32_t own_atoms = static_cast<uint32_t>(4 * half * kAtomBytes);
      bool ok = mbar_wait(Q_FULL, 0) && mbar_wait(Q_TMEM, 0);
      // P V of tile i goes out as soon as the softmax wrote P(i), also between
      // the MMAs of a later tile's Q K^T: it frees the V part that the gather
      // of tile i + 2 waits for, so the gathers do not queue behind the
      // arrival of the next tile.
      int npv = 0;
      auto pv_ready = [&](int nqk) { return npv < nqk && mbar_test_wait(P_FULL, npv & 1); };
      // Descriptors are built once; a K-step adds its compile-time byte
      // offset (>> 4) to the start-address field (addresses stay < 256 KB).
      const uint64_t dstage0 = smem_desc_sw128(sbase + kOffStage, 16, 1024);
      const uint64_t dq = smem_desc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sbase + kOffStage + own_atoms, kAtomBytes, 1024);
      auto issue_pv = [&]() {
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(((npv & 1) * kStageBytes) >> 4);
#pragma unroll
        for (int j = 0; j < kBN / 16; ++j)
          mma_f16_ts(tO, tP + 8 * j, dv + static_cast<uint64_t>((j * 2048) >> 4), idesc_pv,
                     (npv > 0 || j > 0) ? 1u : 0u);
        tc_commit(V_EMPTY(npv & 1));
        tc_commit(PV_DONE);
        ++npv;
      };
// K-step J (compile time) of Q K^T over the stage whose descriptor is DB:
// dims [16 J, 16 J + 16), q from TMEM (J < 20) or shared memory.
#define DSA_QK_STEP(J, DB, ACC)                                                               \
  do {                                                                                       \
    const uint64_t b_ = (DB) + static_cast<uint64_t>(                                        \
                                   ((((J) >> 2) * kAtomBytes) + (((J) & 3) * 32)) >> 4);     \
    if ((J) < kQTmemDims / 16) {                                                             \
      mma_f16_ts(tS, tQ + 8 * (J), b_, idesc_qk, (ACC));                                     \
    } else {                                                                                 \
      const int jq_ = (J) - kQTmemDims / 16;                                                \
      mma_f16_ss(tS, dq + static_cast<uint64_t>(((jq_ >> 2) * kQAtomBytes + (jq_ & 3) * 32) >> 4), \
                 b_, idesc_qk, (ACC));                                                       \
    }                                                                                        \
  } while (0)
      // Waits for a phase while issuing P V as soon as it is ready.
      auto wait_issuing_pv = [&](uint32_t bar, uint32_t parity, int nqk) -> bool {
        const long long t0 = clock64();
        while (!mbar_test_wait(bar, parity)) {
          if (pv_ready(nqk)) issue_pv();
          if (clock64() - t0 > kWaitCycles) return false;
        }
        tc_fence_after();
        return true;
      };
      for (int it = 0; it < ntiles && ok; ++it) {
        const int st = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const uint64_t db = dstage0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
        // Tile it needs the softmax done reading S(it - 1).
        if (it > 0 && !(ok = wait_issuing_pv(S_FREE, (it - 1) & 1, it))) break;
        if constexpr (kFp8) {
          // Dims 0..255 once dequantised, then 256..575.
          if (!(ok = wait_issuing_pv(KV_CONV_A(st), ph, it))) break;
#pragma unroll
          for (int j = 0; j < kLatentDim / 16; ++j) {
            if (j == 16 && !(ok = wait_issuing_pv(KV_CONV(st), ph, it))) break;
            DSA_QK_STEP(j, db, j > 0 ? 1u : 0u);
            if ((j & 7) == 7 && pv_ready(it)) issue_pv();
          }
        } else {
          // The K part (K-steps of the other value half's atoms and of the
          // rope atom), then this CTA's value atoms.
          if (!(ok = wait_issuing_pv(K_FULL(st), ph, it))) break;
          if (half == 0) {
#pragma unroll
            for (int jj = 0; jj < kLatentDim / 16; ++jj) {
              if (jj == 20) {
                tc_commit(K_EMPTY(st));   // freed when the K part's MMAs complete
                if (!(ok = wait_issuing_pv(V_FULL(st), ph, it))) break;
              }
              DSA_QK_STEP(jj < 20 ? 16 + jj : jj - 20, db, jj > 0 ? 1u : 0u);
              if ((jj & 7) == 7 && pv_ready(it)) issue_pv();
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < kLatentDim / 16; ++jj) {
              if (jj == 20) {
                tc_commit(K_EMPTY(st));
                if (!(ok = wait_issuing_pv(V_FULL(st), ph, it))) break;
              }
              DSA_QK_STEP(jj < 16 ? jj : (jj < 20 ? 16 + jj : jj - 4), db, jj > 0 ? 1u : 0u);
              if ((jj & 7) == 7 && pv_ready(it)) issue_pv();
            }
          }
        }
#undef DSA_QK_STEP
        if (!ok) break;
        tc_commit(S_FULL);
      }
      while (ok && npv < ntiles) {
        if (!mbar_wait(P_FULL, npv & 1)) {
          ok = false;
          break;
        }
        issue_pv();
      }
      if (!ok) raise_error(kErrTimeout);
      // Every MMA issued has completed before TMEM is freed.
      tc_commit(MMA_DRAIN);
      mbar_wait(MMA_DRAIN, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Two groups of four warps share the heads: group sg (warps 4-7 or
    // 12-15) owns key columns [32 sg, 32 sg + 32) of each tile, the value
    // dims [128 sg, 128 sg + 128) of the rescale and the epilogue.  A thread
    // and its partner (same head, other group) exchange the tile maximum
    // through shared memory, so both take the same lazy-rescale decision.
    // Every named barrier below is passed once per tile by all 256 threads,
    // also after a failed wait (which only clears `ok`).
    const int sg = warp >> 3;
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t lanebase = static_cast<uint32_t>(q4 * 32) << 16;
    const bool live = h < H;
    bool ok = true;
    // q dims [0, 320) -> TMEM columns [kColQ, kColQ + 160): dims [0, 256)
    // from the TMA copy in stage 1 (row h of each 128B-swizzled atom; group
    // sg moves atoms 2 sg and 2 sg + 1), dims [256, 320) loaded by group 1.
    {
      uint4 qv[8];
      if (sg == 1) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<long long>(t) * H + (live ? h : 0)) * kLatentDim) +
            kQStageAtoms * 8;
#pragma unroll
        for (int u = 0; u < 8; ++u) qv[u] = live ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!mbar_wait(Q_STAGE, 0)) ok = false;
      const uint8_t* qs = smem + kOffStage + kStageBytes + h * 128;
#pragma unroll 1
      for (int c = 2 * sg; c < 2 * sg + 2; ++c) {
        uint32_t rr[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(qs + c * kQAtomBytes + ((u ^ (h & 7)) << 4));
          rr[4 * u + 0] = v.x;
          rr[4 * u + 1] = v.y;
          rr[4 * u + 2] = v.z;
          rr[4 * u + 3] = v.w;
        }
        tmem_st32(tmem + lanebase + kColQ + 32 * c, rr);
      }
      if (sg == 1) {
        uint32_t rr[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          rr[4 * u + 0] = qv[u].x;
          rr[4 * u + 1] = qv[u].y;
          rr[4 * u + 2] = qv[u].z;
          rr[4 * u + 3] = qv[u].w;
        }
        tmem_st32(tmem + lanebase + kColQ + 32 * kQStageAtoms, rr);
      }
      tc_fence_before();
      mbar_arrive(Q_TMEM);
    }
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);   // [2 parities][2 groups][128 heads]
    const float sc = p.sm_scale * 1.4426950408889634f;  // exp -> exp2
    float mrun = ninf, lrun = 0.f;
    for (int it = 0; it < ntiles; ++it) {
      if (ok && !mbar_wait(S_FULL, it & 1)) ok = false;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(tmem + lanebase + kColS + 32 * sg, sr);
      tc_fence_before();
      mbar_arrive(S_FREE);
      const uint32_t msk = mask_s[2 * it + sg];
      float x[32];
      float tmax = ninf;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = ((msk >> j) & 1u) ? __uint_as_float(sr[j]) * sc : ninf;
        tmax = fmaxf(tmax, x[j]);
      }
      // Tile maximum of the head over both groups' columns.
      xchg[((it & 1) * 2 + sg) * 128 + h] = tmax;
      named_bar_sync(3, kSoftThreads);
      tmax = fmaxf(tmax, xchg[((it & 1) * 2 + (sg ^ 1)) * 128 + h]);
      if (it >= 1 && ok && !mbar_wait(PV_DONE, (it - 1) & 1)) ok = false;
      tc_fence_after();
      const bool raise = tmax > mrun + kRescaleLog2;
      const float mnew = raise ? tmax : mrun;
      // O holds a partial sum under the old maximum: rescale this group's
      // half of it (warp-wide, since TMEM loads and stores are warp-collective).
      const bool need = raise && mrun > ninf;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? exp2f(mrun - mnew) : 1.f;
#pragma unroll 1
        for (int c = 4 * sg; c < 4 * sg + 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lanebase + kColO + 32 * c, o);
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * f);
          tmem_st32(tmem + lanebase + kColO + 32 * c, o);
        }
        lrun *= f;
      }
      mrun = mnew;
      uint32_t pk[16];
      float ls = 0.f;
      const bool any = mrun > ninf;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float p0 = any ? exp2f(x[2 * jj] - mrun) : 0.f;
        const float p1 = any ? exp2f(x[2 * jj + 1] - mrun) : 0.f;
        pk[jj] = pack_bf16x2(p0, p1);
        ls += bf16lo_to_f32(pk[jj]) + bf16hi_to_f32(pk[jj]);
      }
      lrun += ls;
      tmem_st16(tmem + lanebase + kColP + 16 * sg, pk);
      tc_fence_before();
      mbar_arrive(P_FULL);
    }
    if (ok && !mbar_wait(PV_DONE, (ntiles - 1) & 1)) ok = false;
    tc_fence_after();
    // Row sum over both groups' columns (parity slot 0 or 1 is free again:
    // both groups passed the last tile's barrier after reading it).
    float* lx = xchg + (ntiles & 1) * 256;
    lx[sg * 128 + h] = ok ? lrun : -1.f;
    named_bar_sync(3, kSoftThreads);
    const float lo = lx[(sg ^ 1) * 128 + h];
    ok = ok && lo >= 0.f;
    const float ltot = lrun + lo;
    if (!ok) raise_error(kErrTimeout);
    // epilogue: O / l -> Mid_O, log-sum-exp -> Mid_LSE.  Each warp owns 32
    // heads and its group's four 32-column chunks; per chunk it stages its
    // 32 x 128 B box in shared memory (the key stages are idle once the last
    // P V is done), 128B-swizzled so that eight consecutive rows' 16-byte
    // stores hit distinct banks, and one lane writes the box with a tensor
    // store (rows past H are clipped).  One TMA instruction per 4 KB instead
    // of one per thread and 1 KB: the copy engine takes a warp's TMA
    // instructions one lane at a time.
    const float inv = (ok && ltot > 0.f) ? 1.f / ltot : 0.f;
    const bool warp_live = q4 * 32 < H;
    const uint32_t box0 = sbase + kOffStage + static_cast<uint32_t>(q4) * kOBoxBytes;
    uint8_t* box0_p = smem + kOffStage + q4 * kOBoxBytes;
#pragma unroll 1
    for (int c = 4 * sg; c < 4 * sg + 4; ++c) {
      uint32_t o[32];
      tmem_ld32(tmem + lanebase + kColO + 32 * c, o);
      uint8_t* row_p = box0_p + c * kOChunkBytes + lane * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<float4*>(row_p + ((u ^ (lane & 7)) << 4)) =
            make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                        __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
      fence_proxy_async_smem();   // generic-proxy writes -> tensor-store reads
      __syncwarp();
      if (warp_live && lane == 0) {
        tma_store_4d(&tmap_o, box0 + c * kOChunkBytes, 256 * half + 32 * c, split, q4 * 32, t);
        bulk_commit();
      }
    }
    if (warp_live && lane == 0) bulk_wait_read_all();
    if (live && half == 0 && sg == 0)
      p.mid_lse[(static_cast<long long>(t) * H + h) * S + split] =
          (ok && ltot > 0.f) ? (mrun + log2f(ltot)) * 0.6931471805599453f : ninf;
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // A selection read without waiting: the grid still completes only after
  // the kernel it depends on (what follows in the stream relies on that).
  if (p.pdl && p.sel_ready && threadIdx.x == 0) grid_dep_wait();
#undef K_FULL
#undef V_FULL
#undef K_EMPTY
#undef V_EMPTY
#undef KV_CONV_A
#undef KV_CONV
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaLaunch& a, cudaStream_t stream) {
  const bool fp8 = a.kv8 != nullptr;
  CUtensorMap tq, tkv, tsc, trope;
  const uint64_t qrows = static_cast<uint64_t>(a.batch) * a.nq * a.heads;
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_pages) * kPage;
  if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kLatentDim, qrows,
                      kLatentDim * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (fp8) {
    // The FP8 rows as bytes: plain 256-byte boxes (codes), 128B-swizzled
    // 128-byte boxes (the rope dims, laid out like a bf16 atom) and 16-byte
    // boxes (the scales).
    if (!encode_tmap_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kv8, kF8RowBytes, cache_rows,
                        kF8RowBytes, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&trope, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kv8, kF8RowBytes, cache_rows,
                        kF8RowBytes, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tsc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kv8, kF8RowBytes, cache_rows,
                        kF8RowBytes, 16, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    // One latent row per box row; gather4 takes four row coordinates per copy.
    if (!encode_tmap_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kv, kLatentDim, cache_rows,
                        kLatentDim * 2, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    tsc = tkv;
    trope = tkv;
  }
  // Mid_O [T][H][S][512] fp32 as a 4-D map; a box is 32 dims x 1 split x 32
  // heads x 1 row, 128B-swizzled.
  CUtensorMap to;
  {
    const uint64_t T = static_cast<uint64_t>(a.batch) * a.nq, S = a.num_splits, H = a.heads;
    const uint64_t dims[4] = {kVDim, S, H, T};
    const uint64_t strides[3] = {kVDim * 4, S * kVDim * 4, H * S * kVDim * 4};
    const uint32_t box[4] = {32, 1, 32, 1};
    if (!encode_tmap_nd(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.mid_o, 4, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  dim3 grid(2 * a.num_splits, a.batch * a.nq);
  // Rows are taken longest first only when the CTAs come in several waves.
  const bool rank = static_cast<long long>(grid.x) * grid.y > device_sm_count();
  auto kern = fp8 ? (rank ? sparse_mla_kernel<true, true> : sparse_mla_kernel<true, false>)
                  : (rank ? sparse_mla_kernel<false, true> : sparse_mla_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, grid, dim3(kThreads), kSmemBytes, stream, a.pdl != 0, 1, tq, tkv, to,
                       tsc, trope, a);
}

}  // namespace dsa
