// fp32 packed varlen attention forward on CUDA cores (FFMA).
//
// The fp32 path must agree with an fp64 reference to 1e-5, which the tf32
// tensor-core rate cannot give, so it runs on the FP32 pipes.  One thread
// block computes a 64-row query tile of one head; each thread owns one query
// row (running max, sum and O row in registers).  KV tiles of 32 keys are
// staged in shared memory and read as broadcasts.  The tile walks its KV runs
// in ring order and folds every KV tile into the running result by exact
// log-sum-exp rescaling ("Scaling video training with parallelism", section 2,
// Ring Attention: blockwise attention over circulating KV blocks).
#include <cmath>

#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

namespace {

constexpr int BM = kSimtTileM;  // 64 query rows
constexpr int BN = kSimtTileN;  // 32 keys

struct SimtParams {
  const float* q;
  const float* k;
  const float* v;
  const QTile* tiles;
  const KvRun* runs;
  void* o;
  float* lse;
  const int64_t* out_map;
  int64_t lse_ld;
  int32_t H, Hkv;
  float scale;
};

template <int D, bool kPartial>
__global__ void __launch_bounds__(BM) attn_fwd_simt_kernel(const SimtParams p) {
  extern __shared__ float simt_smem[];
  float (*sQ)[D + 1] = reinterpret_cast<float (*)[D + 1]>(simt_smem);
  float (*sK)[D] = reinterpret_cast<float (*)[D]>(simt_smem + BM * (D + 1));
  float (*sV)[D] = reinterpret_cast<float (*)[D]>(simt_smem + BM * (D + 1) + BN * D);

  const int tile_id = blockIdx.x / p.H;
  const int h = blockIdx.x - tile_id * p.H;
  const int g = h / (p.H / p.Hkv);
  const QTile tile = p.tiles[tile_id];
  const int row = threadIdx.x;
  const bool valid_row = row < tile.q_rows;
  const int q_pos = tile.q_pos0 + row;

  for (int i = threadIdx.x; i < BM * D; i += BM) {
    const int r = i / D, d = i - r * D;
    sQ[r][d] = (r < tile.q_rows) ? p.q[((int64_t)(tile.q_row0 + r) * p.H + h) * D + d] * p.scale : 0.f;
  }

  float o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int rr = tile.run_begin; rr < tile.run_end; ++rr) {
    const KvRun run = p.runs[rr];
    for (int off = 0; off < run.kv_len; off += BN) {
      const int n_keys = min(BN, run.kv_len - off);
      __syncthreads();
      for (int i = threadIdx.x; i < BN * D; i += BM) {
        const int j = i / D, d = i - j * D;
        const bool in = j < n_keys;
        const int64_t src = ((int64_t)(run.kv_row0 + off + j) * p.Hkv + g) * D + d;
        sK[j][d] = in ? p.k[src] : 0.f;
        sV[j][d] = in ? p.v[src] : 0.f;
      }
      __syncthreads();
      int lim = n_keys;
      if (run.causal) lim = min(lim, q_pos - (run.kv_pos0 + off) + 1);
      float s[BN];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        float acc = 0.f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) acc = fmaf(sQ[row][d], sK[j][d], acc);
        s[j] = (j < lim) ? acc : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      const float m_new = fmaxf(m, mx);
      if (m_new == -INFINITY) continue;  // nothing visible yet for this row
      const float alpha = expf(m - m_new);  // m = -inf gives 0
      l *= alpha;
#pragma unroll
      for (int d = 0; d < D; ++d) o[d] *= alpha;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        const float pj = expf(s[j] - m_new);
        l += pj;
#pragma unroll 16
        for (int d = 0; d < D; ++d) o[d] = fmaf(pj, sV[j][d], o[d]);
      }
      m = m_new;
    }
  }

  if (!valid_row) return;
  const int64_t out_row = p.out_map ? p.out_map[tile.out_row0 + row] : (int64_t)tile.out_row0 + row;
  const bool has = l > 0.f;
  const float inv_l = has ? 1.f / l : 0.f;
  float* dst = static_cast<float*>(p.o) + (out_row * p.H + h) * D;
#pragma unroll
  for (int d = 0; d < D; ++d) dst[d] = has ? o[d] * inv_l : 0.f;
  p.lse[(int64_t)h * p.lse_ld + out_row] = has ? m + logf(l) : -INFINITY;
}

template <int D, bool kPartial>
cudaError_t launch_simt(const SimtParams& p, int64_t blocks, cudaStream_t stream) {
  auto kern = attn_fwd_simt_kernel<D, kPartial>;
  const int smem = (int)sizeof(float) * (BM * (D + 1) + 2 * BN * D);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)blocks, BM, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fp32_simt(const AttnArgs& a, std::string* err) {
  SimtParams p{};
  p.q = static_cast<const float*>(a.q);
  p.k = static_cast<const float*>(a.k);
  p.v = static_cast<const float*>(a.v);
  p.tiles = a.tiles;
  p.runs = a.runs;
  p.o = a.o;
  p.lse = a.lse;
  p.out_map = a.out_map;
  p.lse_ld = a.lse_ld;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.scale = a.scale;
  const int64_t blocks = (int64_t)a.n_tiles * a.H;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) {
    *err = "too many query tiles";
    return cudaErrorInvalidValue;
  }
  if (a.D == 128) return a.partial ? launch_simt<128, true>(p, blocks, a.stream) : launch_simt<128, false>(p, blocks, a.stream);
  return a.partial ? launch_simt<64, true>(p, blocks, a.stream) : launch_simt<64, false>(p, blocks, a.stream);
}

}  // namespace cpattn
