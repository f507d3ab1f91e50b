// dsa_internal.h -- declarations shared by the translation units of libdsa.so
// (launchers and device-error accessors).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct dsa_decode_desc;

namespace dsa {

constexpr int kIndexHeads = 64;
constexpr int kIndexDim = 128;
constexpr int kLatentDim = 576;
constexpr int kVDim = 512;
constexpr int kPage = 64;
constexpr int kHistBins = 2048;     // top 11 bits of the order-preserving score key
constexpr int kHistShift = 21;
constexpr int kTopkChunk = 8192;    // logits per CTA in the top-k passes
constexpr int kTopkClusterCtas = 16;  // CTAs (chunks) per query row in the select pass
// Rows of up to 16 chunks of 4 x 8192 scores.
constexpr int64_t kTopkMaxLd = int64_t(kTopkClusterCtas) * kTopkChunk * 4;

struct IndexerLaunch {
  const uint8_t* q_fp8;
  const float* q_scale;
  const float* w;
  const uint8_t* k_fp8;
  const float* k_scale;
  const int32_t* seqlens;
  const int32_t* page_table;
  float* logits;
  int64_t ld;
  uint32_t* hist;       // [T][kHistBins] or nullptr
  int batch, nq, max_pages, num_pages, topk;
  int skip_short;       // skip requests whose queries all see <= topk tokens
  int pdl;              // 1: launched as a programmatic dependent of the workspace clear
  int wait_tail;        // 1: that kernel also writes new tokens' keys: each request's last
                        //    two tiles are read only after it completed
  long long wait_cycles;   // bound of the pipeline waits (set by launch_indexer)
};

struct TopkLaunch {
  const int32_t* seqlens;
  const float* logits;
  int64_t ld;
  int32_t* out;         // [T][k]
  uint32_t* hist;       // [T][kHistBins], zeroed (or filled by the indexer)
  uint2* cand;          // [T][ld]: chunk c's candidates at the chunk's first position
  int batch, nq, k;
  int hist_ready;       // 1: hist already holds the row histograms
  int pdl;              // 1: launched as a programmatic dependent of the indexer
};

struct CacheWriteLaunch {
  const uint16_t* new_latent;    // [T][576] bf16: the new tokens' latent rows
  const uint16_t* new_index_k;   // [T][128] bf16: the new tokens' indexer keys
  uint16_t* kv;                  // [num_pages * 64][576] bf16 latent cache
  uint8_t* k_fp8;                // [num_pages * 64][128] E4M3 indexer-key cache
  float* k_scale;                // [num_pages * 64] its per-token scales
  const int32_t* seqlens;
  const int32_t* page_table;
  int batch, nq, max_pages, num_pages;
  uint4* clear;                  // zero-filled by CTAs of their own, or nullptr
  long long clear_n16;           // its 16-byte words
};

struct MlaLaunch {
  const uint16_t* q;
  const uint16_t* kv;
  const uint8_t* kv8;   // non-null: the latent cache in FP8 rows of 656 bytes (kv unused)
  const int32_t* topk_idx;
  const int32_t* seqlens;
  const int32_t* page_table;
  float* mid_o;
  float* mid_lse;
  int batch, nq, heads, k, max_pages, num_pages, num_splits;
  float sm_scale;
  int pdl;              // 1: launched as a programmatic dependent of the top-k
  int sel_ready;        // 1: topk_idx was complete before the kernel this one depends on
                        //    started (read without waiting); with pdl the grid then
                        //    completes only after that kernel
};

cudaError_t launch_indexer(const IndexerLaunch& a, cudaStream_t s);
// Bound, in SM cycles, of the indexer's pipeline waits on later launches
// (<= 0: the default kWaitCycles).
void set_indexer_wait_cycles(long long cycles);
cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t s);
cudaError_t launch_sparse_mla(const MlaLaunch& a, cudaStream_t s);
cudaError_t launch_cache_write(const CacheWriteLaunch& a, cudaStream_t s);
cudaError_t launch_latent_fp8(const uint16_t* kv, long long rows, uint8_t* kv8, cudaStream_t s);
cudaError_t launch_merge(int rows, int splits, const float* mid_o, const float* mid_lse,
                         float* out, float* out_lse, cudaStream_t s, bool pdl = false);

// Launches `kern` on `s`; with `pdl` as a programmatic dependent of the
// previous kernel of the stream (the kernel then calls grid_dep_wait before it
// reads anything that kernel wrote).
// `cluster_x` > 1 groups consecutive CTAs along x into clusters of that size.
template <typename... Exp, typename... Act>
cudaError_t launch_kernel(void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, int cluster_x, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Act&&>(args)...);
}

// Each translation unit keeps its own device error word; these read and clear
// them (synchronous).  Return 0 or a dsa_status code.
int fetch_error_indexer();
int fetch_error_topk();
int fetch_error_mla();
int fetch_error_merge();
int fetch_error_cache();

// Host helpers (dsa_api.cu).
// The checks every entry point applies to a decode descriptor: a dsa_status.
int check_decode_desc(const ::dsa_decode_desc* d);
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle);
// Rank-r map (r <= 5): dims[0] is contiguous, byte_strides[i] is the stride
// of dimension i + 1; no fill for out-of-range loads, clipped stores.
bool encode_tmap_nd(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                    const uint64_t* dims, const uint64_t* byte_strides, const uint32_t* box,
                    CUtensorMapSwizzle swizzle);
int device_sm_count();

}  // namespace dsa

// Defines the per-TU device error word and its host accessor.
#define DSA_DEFINE_ERROR_WORD(NAME)                                                    \
  namespace dsa {                                                                      \
  static __device__ int g_error_word = 0;                                              \
  __device__ __forceinline__ void raise_error(int code) {                              \
    atomicCAS(&g_error_word, 0, code);                                                 \
  }                                                                                    \
  int fetch_error_##NAME() {                                                           \
    int v = 0, zero = 0;                                                               \
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 4;  \
    if (v != 0) cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));                  \
    return v;                                                                          \
  }                                                                                    \
  }
