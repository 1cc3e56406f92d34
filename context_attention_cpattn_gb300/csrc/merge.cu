// Exact log-sum-exp merge of ring-step partials (HBM-bound).
//
// Ring attention leaves one partial (O_p, lse_p) per KV block ("Scaling video
// training with parallelism", section 2, Ring Attention); combining them
// exactly is M = max lse_p, lse = M + ln sum exp(lse_p - M),
// O = sum exp(lse_p - lse) O_p.  One warp per (row, head), head-major so that
// neighbouring warps read neighbouring LSE entries: lane i reads the lse of
// partials i and i + 32 once, the weights are formed once and broadcast with
// shuffles, and each lane owns D/32 consecutive elements, loading four
// partials' vectors before their multiply-adds.  The grid is a multiple of the
// SM count and strides over (head, row) pairs.
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
  // head-major order: neighbouring warps read neighbouring LSE entries
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += warps) {
    const int h = (int)(w / p.rows);
    const int64_t row = w - (int64_t)h * p.rows;
    const int64_t li_off = (int64_t)h * p.rows + row;
    // lane i holds the lse of partials i and i + 32, read once
    const float l0 = lane < p.n ? p.lse_parts[lane][li_off] : -INFINITY;
    const float l1 = lane + 32 < p.n ? p.lse_parts[lane + 32][li_off] : -INFINITY;
    float mx = fmaxf(l0, l1);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    const bool has = mx != -INFINITY;
    float z = has ? expf(l0 - mx) + expf(l1 - mx) : 0.f;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) z += __shfl_xor_sync(0xffffffffu, z, s);
    const float lse = has ? mx + logf(z) : -INFINITY;
    const float w0 = has ? expf(l0 - lse) : 0.f;  // weight of partial lane (0 for -inf)
    const float w1 = has ? expf(l1 - lse) : 0.f;  // weight of partial lane + 32

    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (has) {
      // four partials' loads in flight before their multiply-adds
      for (int i0 = 0; i0 < p.n; i0 += 4) {
        float x[4][E];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + k;
          if (i < p.n) {
            const float* src = p.o_parts[i] + (row * p.H + h) * D + lane * E;
            if constexpr (E == 4) {
              const float4 v = *reinterpret_cast<const float4*>(src);
              x[k][0] = v.x;
              x[k][1] = v.y;
              x[k][2] = v.z;
              x[k][3] = v.w;
            } else {
              const float2 v = *reinterpret_cast<const float2*>(src);
              x[k][0] = v.x;
              x[k][1] = v.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) x[k][e] = 0.f;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + k;
          const float wk = __shfl_sync(0xffffffffu, i < 32 ? w0 : w1, i & 31);
          if (i < p.n) {
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, x[k][e], acc[e]);
          }
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
