// C ABI of libcpattn: argument checks, workspace layout and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/cpattn.h"
#include "kernels.hpp"
#include "plan.hpp"

using cpattn::KvRun;
using cpattn::QTile;
using cpattn::WorkList;
using cpattn::WsHeader;

namespace {

thread_local std::string g_err;

// Fault-path test settings (cpattn_debug_wait_fault), written into every
// workspace header a call uploads.  Zero: off.
std::atomic<uint32_t> g_test_wait_limit_us{0};
std::atomic<uint32_t> g_test_withhold{0};

cpattn_status_t fail(cpattn_status_t s, const std::string& msg) {
  g_err = msg;
  return s;
}

cpattn_status_t cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e);
  return CPATTN_CUDA_ERROR;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Plans whose forward runs on head-sharded buffers behind a Ulysses all-to-all.
bool head_sharded(int mode) { return mode == CPATTN_MODE_ULYSSES2D || mode == CPATTN_MODE_PAIRED; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct WsLayout {
  size_t tiles = 0, runs = 0, idx = 0, q = 0, k = 0, v = 0, o = 0, lse = 0, total = 0;
};

size_t elem_size(cpattn_dtype_t dt) { return dt == CPATTN_DTYPE_BF16 ? 2 : 4; }

// header | tiles | runs | (GRID2D: index map | Q shards | K shards | V shards)
WsLayout ws_layout(const cpattn_plan_t& p, const WorkList& wl, int H, int Hkv, int D, size_t es) {
  WsLayout L;
  size_t off = CPATTN_WS_HEADER_BYTES;
  L.tiles = off;
  off += align256(wl.tiles.size() * sizeof(QTile));
  L.runs = off;
  off += align256(wl.runs.size() * sizeof(KvRun));
  if (p.mode == CPATTN_MODE_GRID2D || head_sharded(p.mode)) {
    const bool mesh = head_sharded(p.mode);
    L.idx = off;
    off += align256((size_t)p.T * (mesh ? p.split_h : 1) * sizeof(int64_t));
    L.q = off;
    off += align256((size_t)p.T * H * D * es);
    L.k = off;
    off += align256((size_t)p.T * Hkv * D * es);
    L.v = off;
    off += align256((size_t)p.T * Hkv * D * es);
    if (mesh) {  // head-sharded O and LSE before the reverse all-to-all
      L.o = off;
      off += align256((size_t)p.T * H * D * es);
      L.lse = off;
      off += align256((size_t)p.T * H * sizeof(float));
    }
  }
  L.total = off;
  return L;
}

cpattn_status_t check_shape(int H, int Hkv, int D, cpattn_dtype_t dt) {
  if (dt != CPATTN_DTYPE_FP32 && dt != CPATTN_DTYPE_BF16) return fail(CPATTN_UNSUPPORTED, "dtype must be fp32 or bf16");
  if (D != 64 && D != 128) return fail(CPATTN_UNSUPPORTED, "head dim D must be 64 or 128");
  if (H < 1 || Hkv < 1 || H > 256 || Hkv > 256) return fail(CPATTN_INVALID_ARG, "H and Hkv must be in [1, 256]");
  if (H % Hkv != 0) return fail(CPATTN_INVALID_ARG, "H must be a multiple of Hkv");
  return CPATTN_OK;
}

void tile_sizes(cpattn_dtype_t dt, int* tm, int* tn, bool* pair) {
  if (dt == CPATTN_DTYPE_BF16) {
    *tm = cpattn::kTcTileM;
    *tn = cpattn::kTcTileN;
    *pair = cpattn::kTcPair;
  } else {
    *tm = cpattn::kSimtTileM;
    *tn = cpattn::kSimtTileN;
    *pair = cpattn::kSimtPair;
  }
}

// Host staging of a work list (and the plan's index map) in pinned memory,
// so the per-call upload is a true asynchronous copy.  Kept per work list;
// freed with the plan.
struct Pinned {
  void* ptr = nullptr;
  size_t bytes = 0;
};

struct PlanExtras {
  std::map<const WorkList*, Pinned> worklists;
  Pinned index_map;
};

std::mutex g_extras_mu;
std::map<const cpattn_plan_t*, PlanExtras> g_extras;

cpattn_status_t pinned_copy(const void* src, size_t bytes, Pinned* out) {
  if (out->ptr) return CPATTN_OK;
  if (bytes == 0) return CPATTN_OK;
  cudaError_t e = cudaMallocHost(&out->ptr, bytes);
  if (e != cudaSuccess) {
    out->ptr = nullptr;
    return cuda_fail(e, "cudaMallocHost (work-list staging)");
  }
  memcpy(out->ptr, src, bytes);
  out->bytes = bytes;
  return CPATTN_OK;
}

// Upload the work list (tiles then runs, at their workspace offsets) and clear the fault word.
cpattn_status_t upload_worklist(const cpattn_plan_t* plan, const WorkList& wl, const WsLayout& L, uint8_t* ws,
                                cudaStream_t stream) {
  const size_t tb = wl.tiles.size() * sizeof(QTile), rb = wl.runs.size() * sizeof(KvRun);
  Pinned pt;
  {
    std::lock_guard<std::mutex> lock(g_extras_mu);
    Pinned& slot = g_extras[plan].worklists[&wl];
    if (!slot.ptr && tb + rb > 0) {
      std::vector<uint8_t> buf(L.runs - L.tiles + rb);
      if (tb) memcpy(buf.data(), wl.tiles.data(), tb);
      if (rb) memcpy(buf.data() + (L.runs - L.tiles), wl.runs.data(), rb);
      cpattn_status_t s = pinned_copy(buf.data(), buf.size(), &slot);
      if (s != CPATTN_OK) return s;
    }
    pt = slot;
  }
  cudaError_t e = cudaMemsetAsync(ws, 0, CPATTN_WS_HEADER_BYTES, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (fault word)");
  const uint32_t test_fields[2] = {g_test_wait_limit_us.load(), g_test_withhold.load()};
  if (test_fields[0] || test_fields[1]) {
    // pageable source: the copy is staged before the call returns
    e = cudaMemcpyAsync(ws + offsetof(WsHeader, wait_limit_us), test_fields, sizeof(test_fields),
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (fault-path test settings)");
  }
  if (pt.ptr) {
    e = cudaMemcpyAsync(ws + L.tiles, pt.ptr, pt.bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (work list)");
  }
  return CPATTN_OK;
}

cpattn_status_t upload_index_map(const cpattn_plan_t* plan, uint8_t* dst, cudaStream_t stream) {
  Pinned pm;
  {
    std::lock_guard<std::mutex> lock(g_extras_mu);
    Pinned& slot = g_extras[plan].index_map;
    // GRID2D: the index map; ULYSSES2D: the all-to-all gather map
    const std::vector<int64_t>& m = head_sharded(plan->mode) ? plan->a2a_map : plan->index_map;
    cpattn_status_t s = pinned_copy(m.data(), m.size() * sizeof(int64_t), &slot);
    if (s != CPATTN_OK) return s;
    pm = slot;
  }
  cudaError_t e = cudaMemcpyAsync(dst, pm.ptr, pm.bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (index map)");
  return CPATTN_OK;
}

cpattn_status_t launch_attention(cpattn::AttnArgs& a, cpattn_dtype_t dt) {
  std::string err;
  cudaError_t e = (dt == CPATTN_DTYPE_BF16) ? cpattn::launch_attn_bf16_tc(a, &err) : cpattn::launch_attn_fp32_simt(a, &err);
  if (e != cudaSuccess) {
    if (!err.empty()) return fail(CPATTN_INVALID_ARG, err);
    return cuda_fail(e, "attention kernel launch");
  }
  return CPATTN_OK;
}

// Common checks and setup for cpattn_fwd / cpattn_block_fwd.
cpattn_status_t prepare(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                        cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, int32_t causal, void* ws,
                        size_t ws_bytes) {
  if (!plan) return fail(CPATTN_INVALID_ARG, "plan is NULL");
  cpattn_status_t s = check_shape(H, Hkv, D, dtype);
  if (s != CPATTN_OK) return s;
  if (!q || !k || !v) return fail(CPATTN_INVALID_ARG, "q, k and v must be device pointers");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return fail(CPATTN_INVALID_ARG, "q, k, v must be 16-byte aligned");
  if (causal && plan->mode == CPATTN_MODE_GRID2D)
    return fail(CPATTN_UNSUPPORTED, "causal masks are not defined for grid2d plans");
  if (plan->mode == CPATTN_MODE_PAIRED && !causal)
    return fail(CPATTN_UNSUPPORTED, "paired plans apply the teacher-forcing mask (causal must be 1)");
  if (head_sharded(plan->mode)) {
    if (H % plan->split_h != 0 || Hkv % plan->split_h != 0)
      return fail(CPATTN_UNSUPPORTED, "the Ulysses degree must divide H and Hkv");
    if ((int64_t)plan->T * plan->split_h >= (int64_t(1) << 31))
      return fail(CPATTN_UNSUPPORTED, "u*T must be below 2^31");
  }
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return fail(CPATTN_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
  (void)ws_bytes;
  return CPATTN_OK;
}

// Backward workspace: header | tiles | runs | -lse*log2(e) [H,T] | -delta [H,T] |
// dQ accumulator fp32 [T,H,D] | (GRID2D: index map | Q | K | V | dO shards)
struct BwdLayout {
  size_t tiles = 0, runs = 0, nl2 = 0, nd = 0, dq = 0, idx = 0, q = 0, k = 0, v = 0, dout = 0, total = 0;
};

BwdLayout bwd_layout(const cpattn_plan_t& p, const WorkList& wl, int H, int Hkv, int D, size_t es) {
  BwdLayout L;
  size_t off = CPATTN_WS_HEADER_BYTES;
  L.tiles = off;
  off += align256(wl.tiles.size() * sizeof(QTile));
  L.runs = off;
  off += align256(wl.runs.size() * sizeof(KvRun));
  L.nl2 = off;
  off += align256((size_t)p.T * H * sizeof(float));
  L.nd = off;
  off += align256((size_t)p.T * H * sizeof(float));
  L.dq = off;
  off += align256((size_t)p.T * H * D * sizeof(float));
  if (p.mode == CPATTN_MODE_GRID2D) {
    L.idx = off;
    off += align256((size_t)p.T * sizeof(int64_t));
    L.q = off;
    off += align256((size_t)p.T * H * D * es);
    L.k = off;
    off += align256((size_t)p.T * Hkv * D * es);
    L.v = off;
    off += align256((size_t)p.T * Hkv * D * es);
    L.dout = off;
    off += align256((size_t)p.T * H * D * es);
  }
  L.total = off;
  return L;
}

void bwd_tile_sizes(cpattn_dtype_t dt, int* tk, int* tq) {
  if (dt == CPATTN_DTYPE_BF16) {
    *tk = cpattn::kBwdTcTileK;
    *tq = cpattn::kBwdTcTileQ;
  } else {
    *tk = cpattn::kBwdSimtTileK;
    *tq = cpattn::kBwdSimtTileQ;
  }
}

cpattn_status_t check_bwd_shape(int D, cpattn_dtype_t dt) {
  if (dt == CPATTN_DTYPE_BF16 && D != 128)
    return fail(CPATTN_UNSUPPORTED, "the bf16 backward supports head dim D = 128 (fp32: 64 or 128)");
  return CPATTN_OK;
}

}  // namespace

namespace cpattn {
// Records the message of a failure for cpattn_last_error_string (used by
// entry points defined in other translation units).
cpattn_status_t set_error(cpattn_status_t s, const std::string& msg) { return fail(s, msg); }
}  // namespace cpattn

extern "C" {

cpattn_status_t cpattn_plan(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t cp_size, cpattn_mode_t mode,
                            const cpattn_grid_t* grid, cpattn_plan_t** out_plan) {
  if (!out_plan) return fail(CPATTN_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  auto* p = new (std::nothrow) cpattn_plan_t();
  if (!p) return fail(CPATTN_INVALID_ARG, "out of host memory");
  int32_t g[3] = {0, 0, 0};
  if (grid) {
    g[0] = grid->frames;
    g[1] = grid->height;
    g[2] = grid->width;
  }
  std::string err;
  if (head_sharded(mode)) {
    delete p;
    return fail(CPATTN_INVALID_ARG, "ulysses2d and paired plans are made by cpattn_plan_2d / cpattn_plan_paired");
  }
  try {
    err = cpattn::build_plan(cu_seqlens_host, n_seqs, cp_size, (int32_t)mode, grid ? g : nullptr, p);
  } catch (const std::exception& ex) {
    err = std::string("planner failed: ") + ex.what();
  }
  if (!err.empty()) {
    delete p;
    return fail(CPATTN_INVALID_ARG, err);
  }
  *out_plan = p;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_2d(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t ulysses, int32_t ring,
                               cpattn_plan_t** out_plan) {
  if (!out_plan) return fail(CPATTN_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (ulysses < 1 || ring < 1 || (int64_t)ulysses * ring > 4096)
    return fail(CPATTN_INVALID_ARG, "ulysses and ring must be >= 1 with ulysses*ring <= 4096");
  auto* p = new (std::nothrow) cpattn_plan_t();
  if (!p) return fail(CPATTN_INVALID_ARG, "out of host memory");
  const int32_t g[3] = {ulysses, ring, 0};
  std::string err;
  try {
    err = cpattn::build_plan(cu_seqlens_host, n_seqs, ulysses * ring, CPATTN_MODE_ULYSSES2D, g, p);
  } catch (const std::exception& ex) {
    err = std::string("planner failed: ") + ex.what();
  }
  if (!err.empty()) {
    delete p;
    return fail(CPATTN_INVALID_ARG, err);
  }
  *out_plan = p;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_paired(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t cp_size,
                                   int32_t n_chunks, cpattn_plan_t** out_plan) {
  if (!out_plan) return fail(CPATTN_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (cp_size < 1 || cp_size > 4096) return fail(CPATTN_INVALID_ARG, "cp_size must be in [1, 4096]");
  auto* p = new (std::nothrow) cpattn_plan_t();
  if (!p) return fail(CPATTN_INVALID_ARG, "out of host memory");
  const int32_t g[3] = {n_chunks, 0, 0};
  std::string err;
  try {
    err = cpattn::build_plan(cu_seqlens_host, n_seqs, cp_size, CPATTN_MODE_PAIRED, g, p);
  } catch (const std::exception& ex) {
    err = std::string("planner failed: ") + ex.what();
  }
  if (!err.empty()) {
    delete p;
    return fail(CPATTN_INVALID_ARG, err);
  }
  *out_plan = p;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_allowed_pairs(const cpattn_plan_t* plan, int32_t causal, uint64_t* out) {
  if (!plan || !out) return fail(CPATTN_INVALID_ARG, "NULL argument");
  uint64_t total = 0;
  if (plan->mode == CPATTN_MODE_PAIRED) {
    // clean chunk j sees clean chunks <= j; noisy chunk j sees clean chunks < j and itself
    const int N = plan->tf_chunks;
    for (int s = 0; s < plan->n_seqs; ++s) {
      uint64_t prefix = 0;
      for (int j = 0; j < N; ++j) {
        const uint64_t c = (uint64_t)plan->tf_clean[(size_t)s * N + j].len;
        const uint64_t n = (uint64_t)plan->tf_noisy[(size_t)s * N + j].len;
        total += c * (prefix + c) + n * (prefix + n);
        prefix += c;
      }
    }
  } else {
    for (int s = 0; s < plan->n_seqs; ++s) {
      const uint64_t L = (uint64_t)(plan->cu[s + 1] - plan->cu[s]);
      total += causal ? L * (L + 1) / 2 : L * L;
    }
  }
  *out = total;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_destroy(cpattn_plan_t* plan) {
  if (!plan) return CPATTN_OK;
  {
    std::lock_guard<std::mutex> lock(g_extras_mu);
    auto it = g_extras.find(plan);
    if (it != g_extras.end()) {
      // cudaFreeHost waits for copies that still read the staging buffers
      for (auto& kv : it->second.worklists)
        if (kv.second.ptr) cudaFreeHost(kv.second.ptr);
      if (it->second.index_map.ptr) cudaFreeHost(it->second.index_map.ptr);
      g_extras.erase(it);
    }
  }
  delete plan;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_get_info(const cpattn_plan_t* plan, cpattn_plan_info_t* out) {
  if (!plan || !out) return fail(CPATTN_INVALID_ARG, "NULL argument");
  memset(out, 0, sizeof(*out));
  out->total_tokens = plan->T;
  out->n_chunks = (int64_t)plan->chunk_ranks.size();
  int64_t mx = 0;
  for (int r = 0; r < plan->cp; ++r) mx = std::max<int64_t>(mx, plan->rank_offsets[r + 1] - plan->rank_offsets[r]);
  out->max_rank_tokens = mx;
  out->n_seqs = plan->n_seqs;
  out->cp_size = plan->cp;
  out->mode = plan->mode;
  out->split_h = plan->split_h;
  out->split_w = plan->split_w;
  return CPATTN_OK;
}

#define CPATTN_COPY_OUT(vec)                                                         \
  do {                                                                               \
    if (!plan || !out) return fail(CPATTN_INVALID_ARG, "NULL argument");             \
    if (n < (int64_t)(vec).size()) return fail(CPATTN_INVALID_ARG, "output too small"); \
    if (!(vec).empty()) memcpy(out, (vec).data(), (vec).size() * sizeof((vec)[0]));  \
    return CPATTN_OK;                                                                \
  } while (0)

cpattn_status_t cpattn_plan_get_chunk_offsets(const cpattn_plan_t* plan, int64_t* out, int64_t n) {
  CPATTN_COPY_OUT(plan->chunk_offsets);
}
cpattn_status_t cpattn_plan_get_chunk_ranks(const cpattn_plan_t* plan, int32_t* out, int64_t n) {
  CPATTN_COPY_OUT(plan->chunk_ranks);
}
cpattn_status_t cpattn_plan_get_rank_offsets(const cpattn_plan_t* plan, int64_t* out, int64_t n) {
  CPATTN_COPY_OUT(plan->rank_offsets);
}
cpattn_status_t cpattn_plan_get_index_map(const cpattn_plan_t* plan, int64_t* out, int64_t n) {
  CPATTN_COPY_OUT(plan->index_map);
}

cpattn_status_t cpattn_plan_get_a2a_map(const cpattn_plan_t* plan, int64_t* out, int64_t n) {
  if (plan && !head_sharded(plan->mode)) return fail(CPATTN_INVALID_ARG, "not a ulysses2d or paired plan");
  CPATTN_COPY_OUT(plan->a2a_map);
}

cpattn_status_t cpattn_plan_get_local_cu_seqlens(const cpattn_plan_t* plan, int32_t rank, int32_t* out, int64_t n) {
  if (!plan || !out) return fail(CPATTN_INVALID_ARG, "NULL argument");
  if (rank < 0 || rank >= plan->cp) return fail(CPATTN_INVALID_ARG, "rank out of range");
  if (n < plan->n_seqs + 1) return fail(CPATTN_INVALID_ARG, "output too small");
  memcpy(out, &plan->local_cu[(size_t)rank * (plan->n_seqs + 1)], sizeof(int32_t) * (plan->n_seqs + 1));
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_get_ring_schedule(const cpattn_plan_t* plan, int32_t causal, int32_t* kv_rank,
                                              int32_t* mask_kind, int64_t n) {
  if (!plan || !kv_rank || !mask_kind) return fail(CPATTN_INVALID_ARG, "NULL argument");
  const int cp = plan->cp;
  if (n < (int64_t)cp * cp) return fail(CPATTN_INVALID_ARG, "output too small");
  for (int r = 0; r < cp; ++r)
    for (int t = 0; t < cp; ++t)
      if (!cpattn::ring_entry(*plan, r, t, causal != 0, &kv_rank[r * cp + t], &mask_kind[r * cp + t]))
        return fail(CPATTN_UNSUPPORTED, "causal masks are not defined for grid2d plans");
  return CPATTN_OK;
}

cpattn_status_t cpattn_workspace_size(const cpattn_plan_t* plan, int32_t H, int32_t Hkv, int32_t D,
                                      cpattn_dtype_t dtype, int32_t causal, size_t* bytes) {
  if (!plan || !bytes) return fail(CPATTN_INVALID_ARG, "NULL argument");
  cpattn_status_t s = check_shape(H, Hkv, D, dtype);
  if (s != CPATTN_OK) return s;
  if (causal && plan->mode == CPATTN_MODE_GRID2D)
    return fail(CPATTN_UNSUPPORTED, "causal masks are not defined for grid2d plans");
  int tm, tn;
  bool pair;
  tile_sizes(dtype, &tm, &tn, &pair);
  auto wl = cpattn::get_worklist(*const_cast<cpattn_plan_t*>(plan), causal != 0, tm, tn, pair, -1, 0);
  *bytes = ws_layout(*plan, *wl, H, Hkv, D, elem_size(dtype)).total;
  return CPATTN_OK;
}

cpattn_status_t cpattn_plan_get_worklist(const cpattn_plan_t* cplan, int32_t backward, cpattn_dtype_t dtype,
                                         int32_t causal, int32_t q_rank, int32_t ring_step,
                                         cpattn_work_tile_t* tiles, int64_t max_tiles, cpattn_work_run_t* runs,
                                         int64_t max_runs, int64_t* n_tiles, int64_t* n_runs) {
  if (!cplan || !n_tiles || !n_runs) return fail(CPATTN_INVALID_ARG, "NULL argument");
  if (dtype != CPATTN_DTYPE_FP32 && dtype != CPATTN_DTYPE_BF16) return fail(CPATTN_UNSUPPORTED, "dtype must be fp32 or bf16");
  if (causal && cplan->mode == CPATTN_MODE_GRID2D)
    return fail(CPATTN_UNSUPPORTED, "causal masks are not defined for grid2d plans");
  if (cplan->mode == CPATTN_MODE_PAIRED && !causal)
    return fail(CPATTN_UNSUPPORTED, "paired plans apply the teacher-forcing mask (causal must be 1)");
  if (head_sharded(cplan->mode) && (backward || q_rank >= 0))
    return fail(CPATTN_UNSUPPORTED, "ulysses2d and paired plans run the whole forward only (cpattn_fwd)");
  if (q_rank >= cplan->cp || q_rank < -1) return fail(CPATTN_INVALID_ARG, "q_rank out of range");
  if (q_rank >= 0 && (ring_step < 0 || ring_step >= cplan->cp)) return fail(CPATTN_INVALID_ARG, "ring_step out of range");
  cpattn_plan_t* plan = const_cast<cpattn_plan_t*>(cplan);
  const int step = q_rank >= 0 ? ring_step : 0;
  std::shared_ptr<const WorkList> wl;
  if (backward) {
    int tk, tq;
    bwd_tile_sizes(dtype, &tk, &tq);
    wl = cpattn::get_worklist_bwd(*plan, causal != 0, tk, tq, q_rank, step);
  } else {
    int tm, tn;
    bool pair;
    tile_sizes(dtype, &tm, &tn, &pair);
    wl = cpattn::get_worklist(*plan, causal != 0, tm, tn, pair, q_rank, step);
  }
  *n_tiles = (int64_t)wl->tiles.size();
  *n_runs = (int64_t)wl->runs.size();
  if ((tiles && max_tiles < *n_tiles) || (runs && max_runs < *n_runs))
    return fail(CPATTN_INVALID_ARG, "output too small");
  if (tiles)
    for (size_t i = 0; i < wl->tiles.size(); ++i) {
      const QTile& t = wl->tiles[i];
      tiles[i] = cpattn_work_tile_t{t.q_row0, t.q_pos0, t.out_row0, t.q_rows, t.run_begin, t.run_end, t.n_kv_tiles,
                                    t.rank};
    }
  if (runs)
    for (size_t i = 0; i < wl->runs.size(); ++i) {
      const KvRun& r = wl->runs[i];
      runs[i] = cpattn_work_run_t{r.kv_row0, r.kv_pos0, r.kv_len, r.causal};
    }
  return CPATTN_OK;
}

static cpattn_status_t run_attention(const cpattn_plan_t* cplan, const void* q, const void* k, const void* v,
                                     cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, float scale,
                                     int32_t causal, int q_rank, int step, void* o, float* lse, void* workspace,
                                     size_t ws_bytes, void* stream_ptr) {
  cpattn_status_t s = prepare(cplan, q, k, v, dtype, H, Hkv, D, causal, workspace, ws_bytes);
  if (s != CPATTN_OK) return s;
  if (!o || !lse) return fail(CPATTN_INVALID_ARG, "o and lse must be device pointers");
  if (!aligned16(o)) return fail(CPATTN_INVALID_ARG, "o must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CPATTN_INVALID_ARG, "scale must be positive and finite");
  cpattn_plan_t* plan = const_cast<cpattn_plan_t*>(cplan);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const bool mesh = head_sharded(plan->mode);
  if (mesh && q_rank >= 0)
    return fail(CPATTN_UNSUPPORTED, "ulysses2d and paired plans run the whole forward only (cpattn_fwd)");
  int tm, tn;
  bool pair;
  tile_sizes(dtype, &tm, &tn, &pair);
  // the workspace must hold the whole-forward layout (an upper bound for one step)
  auto wl_all = cpattn::get_worklist(*plan, causal != 0, tm, tn, pair, -1, 0);
  const size_t es = elem_size(dtype);
  const WsLayout L_all = ws_layout(*plan, *wl_all, H, Hkv, D, es);
  if (ws_bytes < L_all.total)
    return fail(CPATTN_WORKSPACE, "workspace too small: need " + std::to_string(L_all.total) + " bytes");
  auto wl = (q_rank < 0) ? wl_all : cpattn::get_worklist(*plan, causal != 0, tm, tn, pair, q_rank, step);
  WsLayout L = ws_layout(*plan, *wl, H, Hkv, D, es);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  s = upload_worklist(plan, *wl, L, ws, stream);
  if (s != CPATTN_OK) return s;

  cpattn::AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.q_rows_total = plan->T;
  a.kv_rows_total = plan->T;
  a.H = H;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.tiles = reinterpret_cast<const QTile*>(ws + L.tiles);
  a.runs = reinterpret_cast<const KvRun*>(ws + L.runs);
  a.n_tiles = (int32_t)wl->tiles.size();
  a.total_pieces = wl->total_kv_tiles;
  a.max_pieces = wl->tiles.empty() ? 0 : wl->tiles.front().n_kv_tiles;  // longest first
  a.o = o;
  a.lse = lse;
  a.ws = reinterpret_cast<WsHeader*>(ws);
  a.stream = stream;
  if (q_rank < 0) {
    a.partial = false;
    a.lse_ld = plan->T;
  } else {
    a.partial = true;
    a.lse_ld = plan->rank_offsets[q_rank + 1] - plan->rank_offsets[q_rank];
  }
  if (mesh) {
    // the all-to-all: rows of (token, head group) gathered into head-sharded buffers
    const int u = plan->split_h;
    const int64_t Hs = H / u, Hks = Hkv / u, R = (int64_t)u * plan->T;
    uint8_t* idx = ws + L_all.idx;
    s = upload_index_map(plan, idx, stream);
    if (s != CPATTN_OK) return s;
    const int64_t* a2a = reinterpret_cast<const int64_t*>(idx);
    cudaError_t e = cpattn::launch_permute_rows(q, ws + L_all.q, a2a, R, Hs * D * es, R, false, stream);
    if (e == cudaSuccess) e = cpattn::launch_permute_rows(k, ws + L_all.k, a2a, R, Hks * D * es, R, false, stream);
    if (e == cudaSuccess) e = cpattn::launch_permute_rows(v, ws + L_all.v, a2a, R, Hks * D * es, R, false, stream);
    if (e != cudaSuccess) return cuda_fail(e, "all-to-all gather");
    a.q = ws + L_all.q;
    a.k = ws + L_all.k;
    a.v = ws + L_all.v;
    a.q_rows_total = a.kv_rows_total = R;
    a.H = (int32_t)Hs;
    a.Hkv = (int32_t)Hks;
    a.o = ws + L_all.o;
    a.lse = reinterpret_cast<float*>(ws + L_all.lse);
    a.lse_ld = R;
    s = launch_attention(a, dtype);
    if (s != CPATTN_OK) return s;
    // the reverse all-to-all of O and LSE
    e = cpattn::launch_permute_rows(ws + L_all.o, o, a2a, R, Hs * D * es, R, true, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_lse_regroup(reinterpret_cast<const float*>(ws + L_all.lse), lse, a2a, (int)Hs, u, plan->T,
                                     stream);
    if (e != cudaSuccess) return cuda_fail(e, "all-to-all scatter");
    return CPATTN_OK;
  }
  if (plan->mode == CPATTN_MODE_GRID2D) {
    // split_cp_2d: gather every rank's shard into contiguous rows
    uint8_t* idx = ws + L_all.idx;
    s = upload_index_map(plan, idx, stream);
    if (s != CPATTN_OK) return s;
    const int64_t* index = reinterpret_cast<const int64_t*>(idx);
    cudaError_t e;
    e = cpattn::launch_permute_rows(q, ws + L_all.q, index, plan->T, (int64_t)H * D * es, plan->T, false, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_permute_rows(k, ws + L_all.k, index, plan->T, (int64_t)Hkv * D * es, plan->T, false, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_permute_rows(v, ws + L_all.v, index, plan->T, (int64_t)Hkv * D * es, plan->T, false, stream);
    if (e != cudaSuccess) return cuda_fail(e, "shard gather");
    a.q = ws + L_all.q;
    a.k = ws + L_all.k;
    a.v = ws + L_all.v;
    // gather_cp_2d: the final outputs go back to global rows through the index map
    if (q_rank < 0) a.out_map = index;
  }
  return launch_attention(a, dtype);
}

cpattn_status_t cpattn_fwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                           cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, float scale, int32_t causal,
                           void* o, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  return run_attention(plan, q, k, v, dtype, H, Hkv, D, scale, causal, -1, 0, o, lse, workspace, ws_bytes, stream);
}

cpattn_status_t cpattn_block_fwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                                 cpattn_dtype_t dtype, int32_t H, int32_t Hkv, int32_t D, float scale, int32_t causal,
                                 int32_t q_rank, int32_t ring_step, float* o_partial, float* lse_partial,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (!plan) return fail(CPATTN_INVALID_ARG, "plan is NULL");
  if (q_rank < 0 || q_rank >= plan->cp) return fail(CPATTN_INVALID_ARG, "q_rank out of range");
  if (ring_step < 0 || ring_step >= plan->cp) return fail(CPATTN_INVALID_ARG, "ring_step out of range");
  return run_attention(plan, q, k, v, dtype, H, Hkv, D, scale, causal, q_rank, ring_step, o_partial, lse_partial,
                       workspace, ws_bytes, stream);
}

cpattn_status_t cpattn_bwd_workspace_size(const cpattn_plan_t* plan, int32_t H, int32_t Hkv, int32_t D,
                                          cpattn_dtype_t dtype, int32_t causal, size_t* bytes) {
  if (!plan || !bytes) return fail(CPATTN_INVALID_ARG, "NULL argument");
  cpattn_status_t s = check_shape(H, Hkv, D, dtype);
  if (s == CPATTN_OK) s = check_bwd_shape(D, dtype);
  if (s != CPATTN_OK) return s;
  if (causal && plan->mode == CPATTN_MODE_GRID2D)
    return fail(CPATTN_UNSUPPORTED, "causal masks are not defined for grid2d plans");
  if (head_sharded(plan->mode)) return fail(CPATTN_UNSUPPORTED, "no backward for ulysses2d or paired plans");
  int tk, tq;
  bwd_tile_sizes(dtype, &tk, &tq);
  auto wl = cpattn::get_worklist_bwd(*const_cast<cpattn_plan_t*>(plan), causal != 0, tk, tq, -1, 0);
  *bytes = bwd_layout(*plan, *wl, H, Hkv, D, elem_size(dtype)).total;
  return CPATTN_OK;
}

static cpattn_status_t run_backward(const cpattn_plan_t* cplan, const void* q, const void* k, const void* v,
                                    const void* o, const float* lse, const void* dout, cpattn_dtype_t dtype,
                                    int32_t H, int32_t Hkv, int32_t D, float scale, int32_t causal, int q_rank,
                                    int step, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                    void* stream_ptr) {
  cpattn_status_t s = prepare(cplan, q, k, v, dtype, H, Hkv, D, causal, workspace, ws_bytes);
  if (s == CPATTN_OK) s = check_bwd_shape(D, dtype);
  if (s != CPATTN_OK) return s;
  if (head_sharded(cplan->mode)) return fail(CPATTN_UNSUPPORTED, "no backward for ulysses2d or paired plans");
  if (!o || !lse || !dout) return fail(CPATTN_INVALID_ARG, "o, lse and dout must be device pointers");
  if (!dq || !dk || !dv) return fail(CPATTN_INVALID_ARG, "dq, dk and dv must be device pointers");
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(CPATTN_INVALID_ARG, "o, dout, dq, dk, dv must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CPATTN_INVALID_ARG, "scale must be positive and finite");
  cpattn_plan_t* plan = const_cast<cpattn_plan_t*>(cplan);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int tk, tq;
  bwd_tile_sizes(dtype, &tk, &tq);
  auto wl_all = cpattn::get_worklist_bwd(*plan, causal != 0, tk, tq, -1, 0);
  const size_t es = elem_size(dtype);
  const BwdLayout L = bwd_layout(*plan, *wl_all, H, Hkv, D, es);
  if (ws_bytes < L.total)
    return fail(CPATTN_WORKSPACE, "workspace too small: need " + std::to_string(L.total) + " bytes");
  auto wl = (q_rank < 0) ? wl_all : cpattn::get_worklist_bwd(*plan, causal != 0, tk, tq, q_rank, step);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsLayout WL;
  WL.tiles = L.tiles;
  WL.runs = L.tiles + align256(wl->tiles.size() * sizeof(QTile));
  s = upload_worklist(plan, *wl, WL, ws, stream);
  if (s != CPATTN_OK) return s;

  cpattn::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout_rows = dout;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.lse_ld = plan->T;
  a.rows_total = plan->T;
  a.H = H;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.bf16 = (dtype == CPATTN_DTYPE_BF16);
  a.tiles = reinterpret_cast<const QTile*>(ws + WL.tiles);
  a.runs = reinterpret_cast<const KvRun*>(ws + WL.runs);
  a.n_tiles = (int32_t)wl->tiles.size();
  a.total_pieces = wl->total_kv_tiles;
  a.max_pieces = wl->tiles.empty() ? 0 : wl->tiles.front().n_kv_tiles;  // longest first
  a.nl2 = reinterpret_cast<float*>(ws + L.nl2);
  a.nd = reinterpret_cast<float*>(ws + L.nd);
  a.ws = reinterpret_cast<WsHeader*>(ws);
  a.stream = stream;
  // dQ accumulates at buffer rows: in the workspace (zeroed by the pre kernel)
  // for the whole backward and for GRID2D steps, directly in the caller's
  // accumulator for the other steps.
  const bool grid2d = (plan->mode == CPATTN_MODE_GRID2D);
  a.accumulate = (q_rank >= 0);
  if (q_rank < 0 || grid2d) {
    a.dq_acc = reinterpret_cast<float*>(ws + L.dq);
    a.zero_dq = true;
  } else {
    a.dq_acc = static_cast<float*>(dq);
    a.zero_dq = false;
  }
  a.dk = dk;
  a.dv = dv;
  if (plan->mode == CPATTN_MODE_GRID2D) {
    // split_cp_2d of Q, K, V and dO; results go back to global rows through the index map
    uint8_t* idx = ws + L.idx;
    s = upload_index_map(plan, idx, stream);
    if (s != CPATTN_OK) return s;
    const int64_t* index = reinterpret_cast<const int64_t*>(idx);
    cudaError_t e;
    e = cpattn::launch_permute_rows(q, ws + L.q, index, plan->T, (int64_t)H * D * es, plan->T, false, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_permute_rows(k, ws + L.k, index, plan->T, (int64_t)Hkv * D * es, plan->T, false, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_permute_rows(v, ws + L.v, index, plan->T, (int64_t)Hkv * D * es, plan->T, false, stream);
    if (e == cudaSuccess)
      e = cpattn::launch_permute_rows(dout, ws + L.dout, index, plan->T, (int64_t)H * D * es, plan->T, false, stream);
    if (e != cudaSuccess) return cuda_fail(e, "shard gather");
    a.q = ws + L.q;
    a.k = ws + L.k;
    a.v = ws + L.v;
    a.dout_rows = ws + L.dout;
    a.in_map = index;
    a.out_map = index;
  }
  cudaError_t e = cpattn::launch_bwd_pre(a);
  if (e != cudaSuccess) return cuda_fail(e, "backward pre kernel");
  std::string err;
  e = a.bf16 ? cpattn::launch_attn_bwd_bf16_tc(a, &err) : cpattn::launch_attn_bwd_fp32_simt(a, &err);
  if (e != cudaSuccess) {
    if (!err.empty()) return fail(CPATTN_INVALID_ARG, err);
    return cuda_fail(e, "backward kernel launch");
  }
  if (q_rank < 0 || grid2d) {
    // whole backward: dQ in the input dtype at global rows; GRID2D step: added to the caller's accumulator
    e = cpattn::launch_bwd_post(a.dq_acc, dq, a.bf16, q_rank >= 0, plan->T, (int64_t)H * D,
                                grid2d ? a.in_map : nullptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward post kernel");
  }
  return CPATTN_OK;
}

cpattn_status_t cpattn_bwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, cpattn_dtype_t dtype, int32_t H, int32_t Hkv,
                           int32_t D, float scale, int32_t causal, void* dq, void* dk, void* dv, void* workspace,
                           size_t ws_bytes, void* stream) {
  return run_backward(plan, q, k, v, o, lse, dout, dtype, H, Hkv, D, scale, causal, -1, 0, dq, dk, dv, workspace,
                      ws_bytes, stream);
}

cpattn_status_t cpattn_block_bwd(const cpattn_plan_t* plan, const void* q, const void* k, const void* v,
                                 const void* o, const float* lse, const void* dout, cpattn_dtype_t dtype, int32_t H,
                                 int32_t Hkv, int32_t D, float scale, int32_t causal, int32_t q_rank,
                                 int32_t ring_step, float* dq_acc, float* dk_acc, float* dv_acc, void* workspace,
                                 size_t ws_bytes, void* stream) {
  if (!plan) return fail(CPATTN_INVALID_ARG, "plan is NULL");
  if (q_rank < 0 || q_rank >= plan->cp) return fail(CPATTN_INVALID_ARG, "q_rank out of range");
  if (ring_step < 0 || ring_step >= plan->cp) return fail(CPATTN_INVALID_ARG, "ring_step out of range");
  return run_backward(plan, q, k, v, o, lse, dout, dtype, H, Hkv, D, scale, causal, q_rank, ring_step, dq_acc,
                      dk_acc, dv_acc, workspace, ws_bytes, stream);
}

cpattn_status_t cpattn_merge(int32_t n_partials, const float* const* o_parts_host, const float* const* lse_parts_host,
                             int64_t rows, int32_t H, int32_t D, const int64_t* out_rows, int64_t out_total_rows,
                             void* o_out, cpattn_dtype_t out_dtype, float* lse_out, void* stream) {
  if (n_partials < 1 || n_partials > 64) return fail(CPATTN_INVALID_ARG, "n_partials must be in [1, 64]");
  if (!o_parts_host || !lse_parts_host || !o_out || !lse_out) return fail(CPATTN_INVALID_ARG, "NULL argument");
  if (D != 64 && D != 128) return fail(CPATTN_UNSUPPORTED, "head dim D must be 64 or 128");
  if (H < 1 || rows < 0) return fail(CPATTN_INVALID_ARG, "bad rows or H");
  if (out_dtype != CPATTN_DTYPE_FP32 && out_dtype != CPATTN_DTYPE_BF16) return fail(CPATTN_UNSUPPORTED, "out dtype");
  if (!out_rows && out_total_rows < rows) return fail(CPATTN_INVALID_ARG, "out_total_rows < rows");
  if (!aligned16(o_out)) return fail(CPATTN_INVALID_ARG, "o_out must be 16-byte aligned");
  cpattn::MergeArgs a;
  a.n = n_partials;
  for (int i = 0; i < n_partials; ++i) {
    if (!o_parts_host[i] || !lse_parts_host[i] || !aligned16(o_parts_host[i]))
      return fail(CPATTN_INVALID_ARG, "partial pointers must be non-NULL, O partials 16-byte aligned");
    a.o_parts[i] = o_parts_host[i];
    a.lse_parts[i] = lse_parts_host[i];
  }
  a.rows = rows;
  a.H = H;
  a.D = D;
  a.out_rows = out_rows;
  a.out_total_rows = out_total_rows;
  a.o_out = o_out;
  a.out_bf16 = out_dtype == CPATTN_DTYPE_BF16;
  a.lse_out = lse_out;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = cpattn::launch_merge(a);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return CPATTN_OK;
}

static cpattn_status_t permute(const void* src, void* dst, const int64_t* index, int64_t rows, int64_t row_bytes,
                               int64_t other_rows, bool scatter, void* stream) {
  if (!src || !dst || (!index && rows > 0)) return fail(CPATTN_INVALID_ARG, "NULL argument");
  if (rows < 0 || other_rows < 0) return fail(CPATTN_INVALID_ARG, "negative row count");
  if (row_bytes <= 0 || (row_bytes & 15)) return fail(CPATTN_INVALID_ARG, "row_bytes must be a positive multiple of 16");
  if (!aligned16(src) || !aligned16(dst)) return fail(CPATTN_INVALID_ARG, "src and dst must be 16-byte aligned");
  cudaError_t e = cpattn::launch_permute_rows(src, dst, index, rows, row_bytes, other_rows, scatter,
                                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "permute kernel launch");
  return CPATTN_OK;
}

cpattn_status_t cpattn_gather_rows(const void* src, int64_t src_rows, void* dst, const int64_t* index, int64_t rows,
                                   int64_t row_bytes, void* stream) {
  return permute(src, dst, index, rows, row_bytes, src_rows, false, stream);
}

cpattn_status_t cpattn_scatter_rows(const void* src, void* dst, int64_t dst_rows, const int64_t* index, int64_t rows,
                                    int64_t row_bytes, void* stream) {
  return permute(src, dst, index, rows, row_bytes, dst_rows, true, stream);
}

cpattn_status_t cpattn_token_loss_norm(const float* loss, const uint8_t* valid, int64_t T, double* out_loss,
                                       int64_t* out_count, float* out_loss_f32, void* stream) {
  if (T < 0) return fail(CPATTN_INVALID_ARG, "T must be >= 0");
  if ((T > 0 && (!loss || !valid)) || !out_loss || !out_count) return fail(CPATTN_INVALID_ARG, "NULL argument");
  cudaError_t e = cpattn::launch_loss_norm(loss, valid, T, out_loss, out_count, out_loss_f32,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "loss kernel launch");
  return CPATTN_OK;
}

cpattn_status_t cpattn_fwd_flops(const int32_t* cu, int32_t n_seqs, int32_t H, int32_t D, int32_t causal,
                                 uint64_t* out_u64, double* out_f64) {
  if (!cu || n_seqs < 1 || H < 1 || D < 1) return fail(CPATTN_INVALID_ARG, "bad arguments");
  unsigned __int128 pairs = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int64_t L = (int64_t)cu[s + 1] - cu[s];
    if (L < 0) return fail(CPATTN_INVALID_ARG, "cu_seqlens must be non-decreasing");
    pairs += causal ? (unsigned __int128)L * (L + 1) / 2 : (unsigned __int128)L * L;
  }
  const unsigned __int128 f = pairs * 4u * (unsigned)D * (unsigned)H;
  if (f > (unsigned __int128)UINT64_MAX) return fail(CPATTN_INVALID_ARG, "FLOP count overflows uint64");
  if (out_u64) *out_u64 = (uint64_t)f;
  if (out_f64) *out_f64 = (double)(uint64_t)f;
  return CPATTN_OK;
}

// Device-side address of a pointer the GPU can reach: device memory as is,
// pinned (registered) host memory through its mapped address; else NULL.
static const void* device_reachable(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return ptr;
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

cpattn_status_t cpattn_copy(void* dst, const void* src, size_t bytes, int32_t n_blocks, void* stream) {
  if (bytes == 0) return CPATTN_OK;
  if (!dst || !src) return fail(CPATTN_INVALID_ARG, "dst and src must not be NULL");
  if ((bytes & 15) || !aligned16(dst) || !aligned16(src))
    return fail(CPATTN_INVALID_ARG, "dst and src must be 16-byte aligned and bytes a multiple of 16");
  const void* s = device_reachable(src);
  void* d = const_cast<void*>(device_reachable(dst));
  if (!s || !d) return fail(CPATTN_INVALID_ARG, "dst and src must be device memory or pinned host memory");
  cudaError_t e = cpattn::launch_copy(s, d, (int64_t)bytes, n_blocks, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy kernel launch");
  return CPATTN_OK;
}

cpattn_status_t cpattn_debug_wait_fault(uint32_t wait_limit_us, int32_t withhold_first_v) {
  if (withhold_first_v != 0 && wait_limit_us == 0)
    return fail(CPATTN_INVALID_ARG, "withholding a load needs a short wait limit (wait_limit_us > 0)");
  if (wait_limit_us > 10000000u) return fail(CPATTN_INVALID_ARG, "wait_limit_us must be at most 10 s");
  g_test_wait_limit_us.store(wait_limit_us);
  g_test_withhold.store(withhold_first_v != 0 ? 1u : 0u);
  return CPATTN_OK;
}

cpattn_status_t cpattn_sync_status(const void* workspace, void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  if (workspace) {
    WsHeader h;
    e = cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the fault word");
    if (h.fault != 0)
      return fail(CPATTN_DEVICE_FAULT, "kernel fault " + std::to_string(h.fault) + " in block " +
                                           std::to_string(h.info) + " at " + std::to_string(h.detail));
  }
  return CPATTN_OK;
}

const char* cpattn_last_error_string(void) { return g_err.c_str(); }

const char* cpattn_version(void) { return "cpattn 0.1.0 (sm_103a)"; }

}  // extern "C"
