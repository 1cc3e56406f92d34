// fp32 packed varlen attention backward on the CUDA cores (the fp32 dtype;
// the bf16 path runs on the tensor cores).  Same work list and same
// arithmetic as the bf16 kernel, in fp32 throughout:
//     P = exp(s - lse), dV += P^T dO, dS = P (dO V^T - delta),
//     dK += scale dS^T Q, dQ += scale dS K
// One block of 128 threads per (KV tile of 32 keys, KV head).  Four threads
// share a key, each holding a quarter of the head dims of its dK and dV rows
// in registers; the block walks the tile's query runs one query (and query
// head) at a time, with the query's Q and dO rows staged in shared memory.
// The query's dQ row is the block-wide sum over keys of dS K, formed in shared
// memory and added to the fp32 accumulator.
#include <cmath>

#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

namespace {

constexpr int kKeys = kBwdSimtTileK;  // 32 keys per block

template <int D>
__global__ void __launch_bounds__(128) attn_bwd_simt_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const QTile* __restrict__ tiles, const KvRun* __restrict__ runs,
    const float* __restrict__ nl2, const float* __restrict__ nd, int64_t ld, float* __restrict__ dq_acc,
    float* __restrict__ dk, float* __restrict__ dv, bool accumulate, const int64_t* __restrict__ out_map,
    int n_tiles, int H, int Hkv, float scale) {
  constexpr int DQ = D / 4;  // head dims per thread
  __shared__ float sK[kKeys][D + 1];
  __shared__ float sq[D], sdo[D];
  __shared__ float sds[kKeys];
  const int tid = threadIdx.x;
  const int key = tid >> 2, part = tid & 3;
  const int item = blockIdx.x;
  const int tile_id = item % n_tiles, g = item / n_tiles;
  const QTile tile = tiles[tile_id];
  const int G = H / Hkv;
  const bool key_ok = key < tile.q_rows;
  const int kp = tile.q_pos0 + key;
  const int64_t krow = (int64_t)tile.q_row0 + (key_ok ? key : 0);

  float kr[DQ], vr[DQ], dkr[DQ], dvr[DQ];
#pragma unroll
  for (int j = 0; j < DQ; ++j) {
    const int d = part * DQ + j;
    kr[j] = key_ok ? k[(krow * Hkv + g) * D + d] : 0.f;
    vr[j] = key_ok ? v[(krow * Hkv + g) * D + d] : 0.f;
    dkr[j] = dvr[j] = 0.f;
  }
  for (int i = tid; i < kKeys * D; i += blockDim.x) {
    const int kk = i / D, d = i % D;
    const bool ok = kk < tile.q_rows;
    sK[kk][d] = ok ? k[(((int64_t)tile.q_row0 + kk) * Hkv + g) * D + d] : 0.f;
  }

  for (int hq = 0; hq < G; ++hq) {
    const int h = g * G + hq;
    for (int r = tile.run_begin; r < tile.run_end; ++r) {
      const KvRun run = runs[r];
      for (int c = 0; c < run.kv_len; ++c) {
        const int64_t qrow = (int64_t)run.kv_row0 + c;
        const int qpos = run.kv_pos0 + c;
        __syncthreads();  // the previous query's rows and dS are consumed
        for (int d = tid; d < D; d += blockDim.x) {
          sq[d] = q[(qrow * H + h) * D + d];
          sdo[d] = dout[(qrow * H + h) * D + d];
        }
        __syncthreads();
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int j = 0; j < DQ; ++j) {
          s = fmaf(sq[part * DQ + j], kr[j], s);
          dp = fmaf(sdo[part * DQ + j], vr[j], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        const float l2 = nl2[(int64_t)h * ld + qrow];
        const bool vis = key_ok && (!run.causal || qpos >= kp) && l2 != -INFINITY;
        const float pr = vis ? exp2f(fmaf(s, scale * 1.4426950408889634f, l2)) : 0.f;
        const float ds = pr * (dp + nd[(int64_t)h * ld + qrow]) * scale;
#pragma unroll
        for (int j = 0; j < DQ; ++j) {
          dvr[j] = fmaf(pr, sdo[part * DQ + j], dvr[j]);
          dkr[j] = fmaf(ds, sq[part * DQ + j], dkr[j]);
        }
        if (part == 0) sds[key] = ds;
        __syncthreads();
        for (int d = tid; d < D; d += blockDim.x) {
          float acc = 0.f;
#pragma unroll 8
          for (int kk = 0; kk < kKeys; ++kk) acc = fmaf(sds[kk], sK[kk][d], acc);
          atomicAdd(dq_acc + (qrow * H + h) * D + d, acc);
        }
      }
    }
  }
  if (!key_ok) return;
  const int64_t orow = out_map ? out_map[krow] : krow;
#pragma unroll
  for (int j = 0; j < DQ; ++j) {
    const int64_t o = (orow * Hkv + g) * D + part * DQ + j;
    if (accumulate) {
      dk[o] += dkr[j];
      dv[o] += dvr[j];
    } else {
      dk[o] = dkr[j];
      dv[o] = dvr[j];
    }
  }
}

}  // namespace

cudaError_t launch_attn_bwd_fp32_simt(const BwdArgs& a, std::string* err) {
  (void)err;
  const int64_t items = (int64_t)a.n_tiles * a.Hkv;
  if (items == 0) return cudaSuccess;
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* d = static_cast<const float*>(a.dout_rows);
  float* dk = static_cast<float*>(a.dk);
  float* dv = static_cast<float*>(a.dv);
  if (a.D == 128)
    attn_bwd_simt_kernel<128><<<(unsigned)items, 128, 0, a.stream>>>(q, k, v, d, a.tiles, a.runs, a.nl2, a.nd,
                                                                     a.rows_total, a.dq_acc, dk, dv, a.accumulate,
                                                                     a.out_map, a.n_tiles, a.H, a.Hkv, a.scale);
  else
    attn_bwd_simt_kernel<64><<<(unsigned)items, 128, 0, a.stream>>>(q, k, v, d, a.tiles, a.runs, a.nl2, a.nd,
                                                                    a.rows_total, a.dq_acc, dk, dv, a.accumulate,
                                                                    a.out_map, a.n_tiles, a.H, a.Hkv, a.scale);
  return cudaGetLastError();
}

}  // namespace cpattn
