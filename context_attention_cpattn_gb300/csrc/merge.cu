// Exact log-sum-exp merge of ring-step partials (HBM-bound).
//
// Ring attention leaves one partial (O_p, lse_p) per KV block ("Scaling video
// training with parallelism", section 2, Ring Attention); combining them
// exactly is M = max lse_p, lse = M + ln sum exp(lse_p - M),
// O = sum exp(lse_p - lse) O_p.  One warp per (row, head): each lane owns D/32
// consecutive elements and reads them with one vector load per partial; the
// per-partial weights are computed once per warp with shuffles.  The grid is a
// multiple of the SM count and strides over (row, head) pairs.
#include <cmath>

#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

namespace {

struct MergeParams {
  const float* o_parts[64];
  const float* lse_parts[64];
  int32_t n;
  int64_t rows;
  int32_t H;
  const int64_t* out_rows;
  int64_t out_total_rows;
  void* o_out;
  float* lse_out;
};

template <int D, bool kBf16>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int E = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t total = p.rows * p.H;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += warps) {
    const int64_t row = w / p.H;
    const int h = (int)(w - row * p.H);
    // max of the partials' lse (each lane takes partials lane, lane+32)
    float mx = -INFINITY;
    for (int i = lane; i < p.n; i += 32) mx = fmaxf(mx, p.lse_parts[i][(int64_t)h * p.rows + row]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    float z = 0.f;
    if (mx != -INFINITY)
      for (int i = lane; i < p.n; i += 32) z += expf(p.lse_parts[i][(int64_t)h * p.rows + row] - mx);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) z += __shfl_xor_sync(0xffffffffu, z, s);
    const bool has = mx != -INFINITY;
    const float lse = has ? mx + logf(z) : -INFINITY;

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (has) {
      for (int i = 0; i < p.n; ++i) {
        const float li = p.lse_parts[i][(int64_t)h * p.rows + row];
        if (li == -INFINITY) continue;
        const float wgt = expf(li - lse);
        const float* src = p.o_parts[i] + (row * p.H + h) * D + lane * E;
        if constexpr (E == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(wgt, x.x, acc[0]);
          acc[1] = fmaf(wgt, x.y, acc[1]);
          acc[2] = fmaf(wgt, x.z, acc[2]);
          acc[3] = fmaf(wgt, x.w, acc[3]);
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(wgt, x.x, acc[0]);
          acc[1] = fmaf(wgt, x.y, acc[1]);
        }
      }
    }
    const int64_t orow = p.out_rows ? p.out_rows[row] : row;
    if (orow < 0 || orow >= p.out_total_rows) continue;
    if constexpr (kBf16) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o_out) + (orow * p.H + h) * D + lane * E;
      if constexpr (E == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(dev::pack_bf16x2(acc[0], acc[1]), dev::pack_bf16x2(acc[2], acc[3]));
      } else {
        *reinterpret_cast<uint32_t*>(dst) = dev::pack_bf16x2(acc[0], acc[1]);
      }
    } else {
      float* dst = static_cast<float*>(p.o_out) + (orow * p.H + h) * D + lane * E;
      if constexpr (E == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
      }
    }
    if (lane == 0) p.lse_out[(int64_t)h * p.out_total_rows + orow] = lse;
  }
}

}  // namespace

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

cudaError_t launch_merge(const MergeArgs& a) {
  MergeParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < a.n; ++i) {
    p.o_parts[i] = a.o_parts[i];
    p.lse_parts[i] = a.lse_parts[i];
  }
  p.n = a.n;
  p.rows = a.rows;
  p.H = a.H;
  p.out_rows = a.out_rows;
  p.out_total_rows = a.out_total_rows;
  p.o_out = a.o_out;
  p.lse_out = a.lse_out;
  const int64_t warps_needed = a.rows * a.H;
  if (warps_needed == 0) return cudaSuccess;
  const int64_t want = (warps_needed + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 8;  // 8 blocks of 8 warps per SM
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  if (a.D == 128) {
    if (a.out_bf16) merge_kernel<128, true><<<blocks, 256, 0, a.stream>>>(p);
    else merge_kernel<128, false><<<blocks, 256, 0, a.stream>>>(p);
  } else {
    if (a.out_bf16) merge_kernel<64, true><<<blocks, 256, 0, a.stream>>>(p);
    else merge_kernel<64, false><<<blocks, 256, 0, a.stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace cpattn
