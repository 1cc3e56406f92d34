// Per-token loss normalisation over valid tokens (Dynamic-CP article,
// section "Loss computation and FLOPS statistics"):
//   loss = sum_t valid_t * loss_t / sum_t valid_t.
// One thread-block cluster of 8 blocks x 1024 threads: each block reads a
// contiguous slice of the fp32 losses and uint8 flags with 16-byte loads and
// accumulates in fp64 / int64 in a fixed stride order; block 0 then adds the
// eight block results, read from the other blocks' shared memory over the
// cluster's distributed shared memory, in rank order.  The result is
// bit-identical from run to run and needs no global scratch.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.hpp"

namespace cg = cooperative_groups;

namespace cpattn {

namespace {

constexpr int kClusterBlocks = 8;

__global__ void __cluster_dims__(kClusterBlocks, 1, 1) __launch_bounds__(1024)
    loss_norm_kernel(const float* __restrict__ loss, const uint8_t* __restrict__ valid, int64_t T,
                     double* out_loss, int64_t* out_count, float* out_f32) {
  __shared__ double s_sum[32];
  __shared__ long long s_cnt[32];
  __shared__ double blk_sum;
  __shared__ long long blk_cnt;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;

  // this block's slice, in whole 16-token groups
  const int64_t groups = (T + 15) / 16;
  const int64_t per = (groups + kClusterBlocks - 1) / kClusterBlocks;
  const int64_t a0 = (int64_t)rank * per * 16, a1 = a0 + per * 16;
  const int64_t t0 = a0 < T ? a0 : T, t1 = a1 < T ? a1 : T;

  double sum = 0.0;
  long long cnt = 0;
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(loss) & 15) == 0) && ((reinterpret_cast<uintptr_t>(valid) & 15) == 0);
  int64_t done = t0;
  if (aligned) {
    // 16 tokens per step: four float4 of losses and one uint4 of flags
    const int64_t n16 = (t1 - t0) / 16;
    const uint4* vf = reinterpret_cast<const uint4*>(valid + t0);
    const float4* lf = reinterpret_cast<const float4*>(loss + t0);
    for (int64_t i = tid; i < n16; i += blockDim.x) {
      const uint4 f = vf[i];
      const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = lf[4 * i + q];
        const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool ok = ((fw[q] >> (8 * e)) & 0xffu) != 0;
          sum += ok ? (double)xv[e] : 0.0;
          cnt += ok ? 1 : 0;
        }
      }
    }
    done = t0 + n16 * 16;
  }
  for (int64_t i = done + tid; i < t1; i += blockDim.x) {
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
      blk_sum = sum;
      blk_cnt = cnt;
    }
  }
  cluster.sync();  // every block's result is in its shared memory
  if (rank == 0 && tid == 0) {
    double total = 0.0;
    long long count = 0;
    for (int r = 0; r < kClusterBlocks; ++r) {
      total += *cluster.map_shared_rank(&blk_sum, r);
      count += *cluster.map_shared_rank(&blk_cnt, r);
    }
    const double v = count > 0 ? total / (double)count : 0.0;
    *out_loss = v;
    *out_count = (int64_t)count;
    if (out_f32) *out_f32 = (float)v;
  }
  cluster.sync();  // keep the blocks (and their shared memory) alive until block 0 has read them
}

}  // namespace

cudaError_t launch_loss_norm(const float* loss, const uint8_t* valid, int64_t T, double* out_loss,
                             int64_t* out_count, float* out_loss_f32, cudaStream_t stream) {
  loss_norm_kernel<<<kClusterBlocks, 1024, 0, stream>>>(loss, valid, T, out_loss, out_count, out_loss_f32);
  return cudaGetLastError();
}

}  // namespace cpattn
