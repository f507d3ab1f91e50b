// merge.cu -- stage 4, the cross-split online-softmax merge ("Deepseek
// Details", section "DSA", stage 3: the blocks' Mid_O and Mid_O_LogExpSum are
// combined into the final output).
//
// One thread per 4 output values of one (query, head) row: it reads the row's
// split log-sum-exps (a broadcast within the row's 128 threads), forms the
// weights exp(lse_b - L) / sum, and streams its 16 bytes of every split's
// partial output with the loads of several splits in flight.
#include "dsa_ptx.cuh"
#include "dsa_internal.h"

DSA_DEFINE_ERROR_WORD(merge)

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = kVDim / 4;   // float4s per row

__global__ void __launch_bounds__(kThreads)
    merge_kernel(int rows, int splits, const float* __restrict__ mid_o,
                 const float* __restrict__ mid_lse, float* __restrict__ out,
                 float* __restrict__ out_lse) {
  grid_dep_wait();   // Mid_O / Mid_LSE may come from the kernel before
  grid_dep_launch();
  const long long gid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const int row = static_cast<int>(gid / kVec);
  const int c4 = static_cast<int>(gid % kVec);
  if (row >= rows) return;
  const float ninf = __int_as_float(0xff800000);
  const float* lse = mid_lse + static_cast<long long>(row) * splits;
  float m = ninf;
  for (int b = 0; b < splits; ++b) m = fmaxf(m, __ldg(lse + b));
  const float4* src = reinterpret_cast<const float4*>(mid_o) +
                      static_cast<long long>(row) * splits * kVec + c4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float tot = 0.f;
  if (m > ninf) {
    // Batches of 8 splits: all loads of a batch are in flight together (an
    // empty split holds zeros and gets weight 0).
    for (int b0 = 0; b0 < splits; b0 += 8) {
      float4 v[8];
      float wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int b = b0 + u;
        if (b < splits) {
          const float l = __ldg(lse + b);
          wv[u] = l > ninf ? __expf(l - m) : 0.f;
          v[u] = __ldg(src + static_cast<long long>(b) * kVec);
        } else {
          wv[u] = 0.f;
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        tot += wv[u];
        acc.x = fmaf(wv[u], v[u].x, acc.x);
        acc.y = fmaf(wv[u], v[u].y, acc.y);
        acc.z = fmaf(wv[u], v[u].z, acc.z);
        acc.w = fmaf(wv[u], v[u].w, acc.w);
      }
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  reinterpret_cast<float4*>(out)[static_cast<long long>(row) * kVec + c4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (out_lse && c4 == 0) out_lse[row] = tot > 0.f ? m + __logf(tot) : ninf;
}

}  // namespace

cudaError_t launch_merge(int rows, int splits, const float* mid_o, const float* mid_lse,
                         float* out, float* out_lse, cudaStream_t stream, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  const long long threads = static_cast<long long>(rows) * kVec;
  const int grid = static_cast<int>((threads + kThreads - 1) / kThreads);
  return launch_kernel(merge_kernel, dim3(grid), dim3(kThreads), 0, stream, pdl, 1, rows, splits,
                       mid_o, mid_lse, out, out_lse);
}

}  // namespace dsa
