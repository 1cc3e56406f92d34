// Per-token loss normalisation over valid tokens (Dynamic-CP article,
// section "Loss computation and FLOPS statistics"):
//   loss = sum_t valid_t * loss_t / sum_t valid_t.
// One block of 1024 threads reads the fp32 losses and uint8 flags with
// 16-byte loads, accumulates in fp64 / int64 per thread in a fixed stride
// order and reduces in a fixed tree, so the result is bit-identical from run
// to run.  The input is a per-token vector (T * 5 bytes), so one block reading
// at a few hundred GB/s finishes in microseconds for micro-batch sizes.
#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

namespace {

__global__ void __launch_bounds__(1024) loss_norm_kernel(const float* __restrict__ loss,
                                                         const uint8_t* __restrict__ valid, int64_t T,
                                                         double* out_loss, int64_t* out_count, float* out_f32) {
  __shared__ double s_sum[32];
  __shared__ long long s_cnt[32];
  double sum = 0.0;
  long long cnt = 0;
  const int tid = threadIdx.x;
  const bool aligned = ((reinterpret_cast<uintptr_t>(loss) & 15) == 0) && ((reinterpret_cast<uintptr_t>(valid) & 15) == 0);
  int64_t done = 0;
  if (aligned) {
    // 16 tokens per step: four float4 of losses and one uint4 of flags
    const int64_t n16 = T / 16;
    for (int64_t i = tid; i < n16; i += blockDim.x) {
      const uint4 f = reinterpret_cast<const uint4*>(valid)[i];
      const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = reinterpret_cast<const float4*>(loss)[4 * i + q];
        const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool ok = ((fw[q] >> (8 * e)) & 0xffu) != 0;
          sum += ok ? (double)xv[e] : 0.0;
          cnt += ok ? 1 : 0;
        }
      }
    }
    done = n16 * 16;
  }
  for (int64_t i = done + tid; i < T; i += blockDim.x) {
    const bool ok = valid[i] != 0;
    sum += ok ? (double)loss[i] : 0.0;
    cnt += ok ? 1 : 0;
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, s);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, s);
  }
  if ((tid & 31) == 0) {
    s_sum[tid >> 5] = sum;
    s_cnt[tid >> 5] = cnt;
  }
  __syncthreads();
  if (tid < 32) {
    sum = s_sum[tid];
    cnt = s_cnt[tid];
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, s);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, s);
    }
    if (tid == 0) {
      const double v = cnt > 0 ? sum / (double)cnt : 0.0;
      *out_loss = v;
      *out_count = (int64_t)cnt;
      if (out_f32) *out_f32 = (float)v;
    }
  }
}

}  // namespace

cudaError_t launch_loss_norm(const float* loss, const uint8_t* valid, int64_t T, double* out_loss,
                             int64_t* out_count, float* out_loss_f32, cudaStream_t stream) {
  loss_norm_kernel<<<1, 1024, 0, stream>>>(loss, valid, T, out_loss, out_count, out_loss_f32);
  return cudaGetLastError();
}

}  // namespace cpattn
