// cache_write.cu -- the step before the indexer: every new token's latent row
// is written into the paged MLA cache at its position, and its indexer key is
// stored as FP8 E4M3 with one fp32 scale per token ("[SGLang] NSA", section
// "forward_decode": set_mla_kv_buffer before the attention; the module list's
// quant_k_cache, the NSA-specific FP8 quantisation of the K cache; "Sparse
// attention: NSA and DSA": the indexer key, FP8 + scale).
//
// Token i of request r (row t = r * n_q + i) is the request's
// (S_r - n_q + i)-th token: the n_q new tokens are the last of the S_r.  The
// scale is amax / 448 over the token's 128 key values (448: E4M3's largest
// finite magnitude), the codes E4M3(k / scale) rounded to nearest even and
// saturated, all in fp32; a token of zeros gets scale 1 and zero codes.
//
// One warp per new token: the 1152-byte latent row moves as 72 16-byte words;
// each lane holds 4 of the key's 128 values, and a warp-wide maximum gives
// amax.  The work is a few KB: the kernel is launch-bound, so on the fused
// layer it also zero-fills the top-k histogram, in CTAs of its own.
#include <cuda_fp8.h>

#include <algorithm>

#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(cache)

namespace dsa {
namespace {

constexpr int kWarps = 8;   // tokens (rows) per CTA
constexpr int kF8LatentBytes = 656;

// Writes new token t (one warp).
__device__ __forceinline__ void write_token(const CacheWriteLaunch& p, int t, int lane) {
  const int r = t / p.nq, i = t % p.nq;
  const int pos = p.seqlens[r] - p.nq + i;
  if (pos < 0 || pos >= p.max_pages * kPage) {
    if (lane == 0) raise_error(kErrCheck);
    return;
  }
  const int pg = p.page_table[static_cast<long long>(r) * p.max_pages + (pos >> 6)];
  if (pg < 0 || pg >= p.num_pages) {
    if (lane == 0) raise_error(kErrCheck);
    return;
  }
  const long long row = static_cast<long long>(pg) * kPage + (pos & (kPage - 1));

  // The latent row, bit for bit.
  const uint4* src = reinterpret_cast<const uint4*>(p.new_latent + static_cast<long long>(t) * kLatentDim);
  uint4* dst = reinterpret_cast<uint4*>(p.kv + row * kLatentDim);
  for (int c = lane; c < kLatentDim * 2 / 16; c += 32) dst[c] = __ldg(src + c);

  // The indexer key: values 4 lane .. 4 lane + 3.
  const uint2 kb =
      __ldg(reinterpret_cast<const uint2*>(p.new_index_k + static_cast<long long>(t) * kIndexDim) + lane);
  const float k[4] = {bf16lo_to_f32(kb.x), bf16hi_to_f32(kb.x), bf16lo_to_f32(kb.y), bf16hi_to_f32(kb.y)};
  float amax = fmaxf(fmaxf(fabsf(k[0]), fabsf(k[1])), fmaxf(fabsf(k[2]), fabsf(k[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t codes = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    codes |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(k[e] / scale, __NV_SATFINITE, __NV_E4M3))
             << (8 * e);
  reinterpret_cast<uint32_t*>(p.k_fp8 + row * kIndexDim)[lane] = codes;
  if (lane == 0) p.k_scale[row] = scale;
}

// CTAs [0, ceil(T / kWarps)) write the new tokens; the CTAs after them, if
// any, zero-fill p.clear (the layer's top-k histogram).  The kernel lets
// its dependent (the indexer) start at once: that kernel waits for it before
// it reads the new tokens' keys or its first histogram flush.
__global__ void __launch_bounds__(kWarps * 32) cache_write_kernel(const CacheWriteLaunch p) {
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.batch * p.nq;
  const int nw = (T + kWarps - 1) / kWarps;
  if (static_cast<int>(blockIdx.x) < nw) {
    const int t = blockIdx.x * kWarps + warp;
    if (t < T) write_token(p, t, lane);
    return;
  }
  const long long step = static_cast<long long>(gridDim.x - nw) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x - nw) * blockDim.x + threadIdx.x; i < p.clear_n16;
       i += step)
    p.clear[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Latent rows in FP8 (656 bytes: the 512 value dims as four 128-dim tiles of
// E4M3 codes, each with an fp32 scale amax / 448 -- the fine-grained 1 x 128
// tiles of "Deepseek Details", section "FP8 Training" -- then the four
// scales, then the 64 rope dims as bf16).  One warp per row: lane l holds
// dims 16 l .. 16 l + 15 (tile l / 8), eight lanes reduce a tile's amax.
__global__ void __launch_bounds__(kWarps * 32) latent_fp8_kernel(const uint16_t* __restrict__ kv,
                                                                 long long rows,
                                                                 uint8_t* __restrict__ kv8) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(kv + row * kLatentDim);
  const uint4 v0 = __ldg(src + 2 * lane), v1 = __ldg(src + 2 * lane + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[2 * e] = bf16lo_to_f32(w[e]);
    x[2 * e + 1] = bf16hi_to_f32(w[e]);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t codes[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e)
    codes[e >> 2] |=
        static_cast<uint32_t>(__nv_cvt_float_to_fp8(x[e] / scale, __NV_SATFINITE, __NV_E4M3))
        << (8 * (e & 3));
  uint8_t* dst = kv8 + row * kF8LatentBytes;
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  if ((lane & 7) == 0) reinterpret_cast<float*>(dst + 512)[lane >> 3] = scale;
  if (lane < 8)
    reinterpret_cast<uint4*>(dst + 528)[lane] = __ldg(src + (512 * 2) / 16 + lane);
}

}  // namespace

cudaError_t launch_latent_fp8(const uint16_t* kv, long long rows, uint8_t* kv8,
                              cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long grid = (rows + kWarps - 1) / kWarps;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  latent_fp8_kernel<<<dim3(static_cast<unsigned>(grid)), dim3(kWarps * 32), 0, stream>>>(kv, rows,
                                                                                        kv8);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const CacheWriteLaunch& a, cudaStream_t stream) {
  const int T = a.batch * a.nq;
  const int nw = (T + kWarps - 1) / kWarps;
  const long long nc = a.clear_n16 > 0 ? std::min<long long>((a.clear_n16 + 255) / 256, 148) : 0;
  if (nw + nc == 0) return cudaSuccess;
  return launch_kernel(cache_write_kernel, dim3(static_cast<unsigned>(nw + nc)), dim3(kWarps * 32), 0,
                       stream, false, 1, a);
}

}  // namespace dsa
