// merge.cu -- stage 4, the cross-split online-softmax merge ("Deepseek
// Details", section "DSA", stage 3: the blocks' Mid_O and Mid_O_LogExpSum are
// combined into the final output).
//
// One warp per (query, head) row: the lanes hold the splits' log-sum-exps,
// reduce their maximum L and the weights exp(lse_b - L) by shuffles, then
// stream the splits' 512-float partial outputs with 16-byte loads.
#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(merge)

namespace dsa {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    merge_kernel(int rows, int splits, const float* __restrict__ mid_o,
                 const float* __restrict__ mid_lse, float* __restrict__ out,
                 float* __restrict__ out_lse) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float ninf = __int_as_float(0xff800000);
  float lse = lane < splits ? __ldg(mid_lse + static_cast<long long>(row) * splits + lane) : ninf;
  float m = lse;
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const bool empty = !(m > ninf);
  float wgt = (!empty && lse > ninf) ? __expf(lse - m) : 0.f;
  float tot = wgt;
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* src = reinterpret_cast<const float4*>(mid_o + static_cast<long long>(row) * splits * kVDim);
  for (int b = 0; b < splits; ++b) {
    const float wb = __shfl_sync(0xffffffffu, wgt, b) * inv;
    if (wb == 0.f) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldg(src + b * (kVDim / 4) + q * 32 + lane);
      acc[q].x = fmaf(wb, v.x, acc[q].x);
      acc[q].y = fmaf(wb, v.y, acc[q].y);
      acc[q].z = fmaf(wb, v.z, acc[q].z);
      acc[q].w = fmaf(wb, v.w, acc[q].w);
    }
  }
  float4* dst = reinterpret_cast<float4*>(out + static_cast<long long>(row) * kVDim);
#pragma unroll
  for (int q = 0; q < 4; ++q) dst[q * 32 + lane] = acc[q];
  if (out_lse && lane == 0) out_lse[row] = tot > 0.f ? m + __logf(tot) : ninf;
}

}  // namespace

cudaError_t launch_merge(int rows, int splits, const float* mid_o, const float* mid_lse,
                         float* out, float* out_lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + kWarps - 1) / kWarps;
  merge_kernel<<<grid, kWarps * 32, 0, stream>>>(rows, splits, mid_o, mid_lse, out, out_lse);
  return cudaGetLastError();
}

}  // namespace dsa
