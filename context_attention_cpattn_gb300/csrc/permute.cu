// Row permutation between global THD order and per-rank shards: the one-GPU
// equivalents of LongCat-Video's split_cp_2d (scatter pieces to ranks) and
// gather_cp_2d (reassemble them) (LongCat-Video context-parallel article,
// communication primitives).  HBM-bound copy: one warp per row, 16-byte
// vector loads and stores, grid a multiple of the SM count striding over rows.
#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

namespace {

template <bool kScatter>
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const int64_t* __restrict__ index, int64_t rows,
                                                           int64_t row_vecs, int64_t other_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < rows; i += warps) {
    const int64_t j = index[i];
    if (j < 0 || j >= other_rows) continue;  // out-of-range rows are skipped
    const uint4* s = src + (kScatter ? i : j) * row_vecs;
    uint4* d = dst + (kScatter ? j : i) * row_vecs;
    for (int64_t c = lane; c < row_vecs; c += 32) d[c] = s[c];
  }
}

// Reverse all-to-all of the log-sum-exp: the head-sharded buffer holds
// [H/u heads][u*T rows] (row R = i*T + p of head group i); the output is
// [H][T] at global rows.  a2a[R] = t*u + i names the token and head group.
__global__ void __launch_bounds__(256) lse_regroup_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                          const int64_t* __restrict__ a2a, int Hs, int u, int64_t T) {
  const int64_t n = (int64_t)Hs * u * T;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += stride) {
    const int64_t hl = idx / (u * T), R = idx - hl * (u * T);
    const int64_t m = a2a[R];
    const int64_t t = m / u, i = m - t * u;
    dst[(i * Hs + hl) * T + t] = src[idx];
  }
}

// Plain copy of n 16-byte vectors, four loads in flight per thread.  Either
// side may be pinned host memory that the GPU reads or writes over the
// host link (NVLink-C2C on Grace hosts).
__global__ void __launch_bounds__(256) copy_vec_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, int n_blocks, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  const int64_t n = bytes / 16;
  const int64_t want = (n + 255) / 256;
  const int64_t cap = n_blocks > 0 ? n_blocks : (int64_t)num_sms() * 4;
  copy_vec_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, stream>>>(static_cast<const uint4*>(src),
                                                                           static_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_lse_regroup(const float* src, float* dst, const int64_t* a2a, int Hs, int u, int64_t T,
                               cudaStream_t stream) {
  const int64_t n = (int64_t)Hs * u * T;
  if (n == 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256, cap = (int64_t)num_sms() * 16;
  lse_regroup_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, stream>>>(src, dst, a2a, Hs, u, T);
  return cudaGetLastError();
}

cudaError_t launch_permute_rows(const void* src, void* dst, const int64_t* index, int64_t rows, int64_t row_bytes,
                                int64_t other_rows, bool scatter, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t want = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 8;
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  const int64_t vecs = row_bytes / 16;
  if (scatter)
    permute_rows_kernel<true><<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                          index, rows, vecs, other_rows);
  else
    permute_rows_kernel<false><<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                           index, rows, vecs, other_rows);
  return cudaGetLastError();
}

}  // namespace cpattn
