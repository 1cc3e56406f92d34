// Launch descriptors for the CUDA kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "worklist.h"

namespace cpattn {

// One attention launch over a work list.  Q/K/V are [rows, heads, D]
// buffers (global THD tensors, or gathered shards for GRID2D).
struct AttnArgs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t q_rows_total = 0;   // rows in the Q buffer
  int64_t kv_rows_total = 0;  // rows in the K/V buffers
  int32_t H = 0, Hkv = 0, D = 0;
  float scale = 0.f;
  const QTile* tiles = nullptr;  // device
  const KvRun* runs = nullptr;   // device
  int32_t n_tiles = 0;
  int64_t total_pieces = 0;      // KV pieces over all tiles (one head's work)
  int32_t max_pieces = 0;        // KV pieces of the longest tile
  void* o = nullptr;             // final: dtype [*,H,D] at global rows; partial: fp32 [*,H,D]
  bool partial = false;
  float* lse = nullptr;          // [H, lse_ld]
  int64_t lse_ld = 0;
  const int64_t* out_map = nullptr;  // optional: output row = out_map[row]
  WsHeader* ws = nullptr;
  cudaStream_t stream = nullptr;
};

// q tile / KV tile sizes each attention kernel was built for ("pair": two
// consecutive KV pieces form one kernel tile).
constexpr int kTcTileM = 128, kTcTileN = 64;
constexpr bool kTcPair = false;
constexpr int kSimtTileM = 64, kSimtTileN = 32;
constexpr bool kSimtPair = false;

cudaError_t launch_attn_bf16_tc(const AttnArgs& a, std::string* err);
cudaError_t launch_attn_fp32_simt(const AttnArgs& a, std::string* err);

// One backward launch over a backward work list (KV tiles with query runs).
struct BwdArgs {
  const void* q = nullptr;          // rows the kernel reads (gathered shards for GRID2D)
  const void* k = nullptr;
  const void* v = nullptr;
  const void* dout_rows = nullptr;  // dO in the same row order as q
  const void* o = nullptr;          // O and dO at global rows (read by the pre kernel through in_map)
  const void* dout = nullptr;
  const float* lse = nullptr;       // [H, lse_ld] at global rows
  int64_t lse_ld = 0;
  const int64_t* in_map = nullptr;  // buffer row -> global row, or null
  int64_t rows_total = 0;
  int32_t H = 0, Hkv = 0, D = 0;
  float scale = 0.f;
  bool bf16 = true;
  const QTile* tiles = nullptr;     // device
  const KvRun* runs = nullptr;      // device
  int32_t n_tiles = 0;
  int64_t total_pieces = 0;      // query pieces over all KV tiles (one KV head's work per query head)
  int32_t max_pieces = 0;        // query pieces of the longest KV tile
  float* nl2 = nullptr;             // scratch [H, rows_total]: -lse*log2(e)
  float* nd = nullptr;              // scratch [H, rows_total]: -rowsum(dO*O)
  float* dq_acc = nullptr;          // fp32 [rows_total, H, D] at buffer rows, accumulated
  bool zero_dq = false;             // the pre kernel clears dq_acc first
  void* dk = nullptr;               // output dtype [*, Hkv, D] stored, or fp32 accumulated
  void* dv = nullptr;
  bool accumulate = false;
  const int64_t* out_map = nullptr; // output row of a buffer row for dK / dV, or null
  WsHeader* ws = nullptr;
  cudaStream_t stream = nullptr;
};

// Backward tiles: KV tiles of kBwdTileK keys, query pieces of kBwdTileQ.
constexpr int kBwdTcTileK = 128, kBwdTcTileQ = 64;
constexpr int kBwdSimtTileK = 32, kBwdSimtTileQ = 64;

cudaError_t launch_bwd_pre(const BwdArgs& a);
cudaError_t launch_attn_bwd_bf16_tc(const BwdArgs& a, std::string* err);
cudaError_t launch_attn_bwd_fp32_simt(const BwdArgs& a, std::string* err);
// dQ accumulator (fp32, buffer rows of row_elems values) to the output at
// rows map[r] (or r): stored in the output dtype, or added to a fp32 output.
cudaError_t launch_bwd_post(const float* dq_acc, void* out, bool out_bf16, bool add, int64_t rows,
                            int64_t row_elems, const int64_t* map, cudaStream_t stream);

struct MergeArgs {
  int32_t n = 0;
  const float* o_parts[64] = {};
  const float* lse_parts[64] = {};
  int64_t rows = 0;
  int32_t H = 0, D = 0;
  const int64_t* out_rows = nullptr;
  int64_t out_total_rows = 0;
  void* o_out = nullptr;
  bool out_bf16 = false;
  float* lse_out = nullptr;
  cudaStream_t stream = nullptr;
};
cudaError_t launch_merge(const MergeArgs& a);

cudaError_t launch_loss_norm(const float* loss, const uint8_t* valid, int64_t T, double* out_loss,
                             int64_t* out_count, float* out_loss_f32, cudaStream_t stream);

// gather: dst[i] = src[index[i]]; scatter: dst[index[i]] = src[i].  Rows whose
// index falls outside [0, other_rows) are skipped.
cudaError_t launch_permute_rows(const void* src, void* dst, const int64_t* index, int64_t rows,
                                int64_t row_bytes, int64_t other_rows, bool scatter, cudaStream_t stream);

// dst[(i*Hs + h)*T + t] = src[h*(u*T) + R] with a2a[R] = t*u + i (the reverse
// all-to-all of a head-sharded LSE buffer).
cudaError_t launch_lse_regroup(const float* src, float* dst, const int64_t* a2a, int Hs, int u, int64_t T,
                               cudaStream_t stream);

// dst[0, bytes) = src[0, bytes): 16-byte aligned, bytes a multiple of 16;
// either pointer may be pinned host memory the device can address.
// n_blocks <= 0: four blocks per SM.
cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, int n_blocks, cudaStream_t stream);

int num_sms();

// TMA tensor maps of a [rows, heads, D] tensor viewed as (D, heads, rows):
// bf16 with 64-column boxes and 128-byte swizzle, or fp32 with D-column boxes
// and no swizzle.  On failure *err says why.
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows,
                          std::string* err);
bool make_tensor_map_f32(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows,
                         std::string* err);

}  // namespace cpattn
