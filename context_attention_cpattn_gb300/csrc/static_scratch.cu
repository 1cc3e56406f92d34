// Workspace-free packed forward: cpattn_fwd_static.
//
// Some callers cannot allocate device memory for the library at all: a
// plugin or custom-operator interface that hands over only the input and
// output buffers, or a process whose device memory is owned entirely by
// another allocator that the caller cannot ask for scratch.  For them this
// entry point runs the same packed forward as cpattn_fwd, but keeps its
// scratch (the fault word and the uploaded work list) in a fixed array that
// lives in the library's own device image, so it allocates nothing.
//
// The array is CPATTN_STATIC_SCRATCH_BYTES (8 MiB) on every GPU that loads
// the library, held until the process exits.  Host code cannot use the
// array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// caches it.  A kernel that gives up on a bounded wait records the fault in
// the array's header; cpattn_static_sync_status reads it back (again without
// allocating).
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/cpattn.h"
#include "kernels.hpp"
#include "plan.hpp"

namespace cpattn {
cpattn_status_t set_error(cpattn_status_t s, const std::string& msg);  // api.cpp
}

static __device__ __align__(256) uint8_t g_cpattn_static_scratch[CPATTN_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the static scratch on the current device (looked up once per device).
cpattn_status_t scratch_on_current_device(uint8_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cpattn::set_error(CPATTN_CUDA_ERROR, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return cpattn::set_error(CPATTN_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_cpattn_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return cpattn::set_error(CPATTN_CUDA_ERROR,
                               std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return CPATTN_OK;
}

}  // namespace

extern "C" cpattn_status_t cpattn_fwd_static(const cpattn_plan_t* cplan, const void* q, const void* k,
                                             const void* v, cpattn_dtype_t dtype, int32_t H, int32_t Hkv,
                                             int32_t D, float scale, int32_t causal, void* o, float* lse,
                                             void* stream_ptr) {
  using cpattn::set_error;
  if (!cplan) return set_error(CPATTN_INVALID_ARG, "plan is NULL");
  if (dtype != CPATTN_DTYPE_FP32 && dtype != CPATTN_DTYPE_BF16) return set_error(CPATTN_UNSUPPORTED, "dtype must be fp32 or bf16");
  if (D != 64 && D != 128) return set_error(CPATTN_UNSUPPORTED, "head dim D must be 64 or 128");
  if (H < 1 || Hkv < 1 || H > 256 || Hkv > 256 || H % Hkv != 0)
    return set_error(CPATTN_INVALID_ARG, "H and Hkv must be in [1, 256] with H a multiple of Hkv");
  if (!q || !k || !v || !o || !lse) return set_error(CPATTN_INVALID_ARG, "q, k, v, o and lse must be device pointers");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if (mis & 15) return set_error(CPATTN_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return set_error(CPATTN_INVALID_ARG, "scale must be positive and finite");
  if (cplan->mode == CPATTN_MODE_GRID2D || cplan->mode == CPATTN_MODE_ULYSSES2D ||
      cplan->mode == CPATTN_MODE_PAIRED)
    return set_error(CPATTN_UNSUPPORTED,
                     "cpattn_fwd_static has no room to gather grid2d, ulysses2d or paired shards; use cpattn_fwd "
                     "with a workspace");

  cpattn_plan_t* plan = const_cast<cpattn_plan_t*>(cplan);
  const bool bf16 = dtype == CPATTN_DTYPE_BF16;
  const int tm = bf16 ? cpattn::kTcTileM : cpattn::kSimtTileM, tn = bf16 ? cpattn::kTcTileN : cpattn::kSimtTileN;
  const bool pair = bf16 ? cpattn::kTcPair : cpattn::kSimtPair;
  auto wl = cpattn::get_worklist(*plan, causal != 0, tm, tn, pair, -1, 0);
  const size_t tb = wl->tiles.size() * sizeof(cpattn::QTile), rb = wl->runs.size() * sizeof(cpattn::KvRun);
  const size_t off_tiles = CPATTN_WS_HEADER_BYTES, off_runs = off_tiles + round256(tb);
  const size_t need = off_runs + round256(rb);
  if (need > CPATTN_STATIC_SCRATCH_BYTES)
    return set_error(CPATTN_WORKSPACE, "the work list needs " + std::to_string(need) +
                                           " bytes but the static scratch holds " +
                                           std::to_string((size_t)CPATTN_STATIC_SCRATCH_BYTES) +
                                           "; use cpattn_fwd with a workspace");
  uint8_t* base = nullptr;
  cpattn_status_t s = scratch_on_current_device(&base);
  if (s != CPATTN_OK) return s;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  // The scratch keeps the previous call's contents: clear the fault word, then
  // overwrite the work list (from the plan's host copy; pageable, so these
  // copies are staged by the driver before the call returns).
  cudaError_t e = cudaMemsetAsync(base, 0, CPATTN_WS_HEADER_BYTES, stream);
  if (e == cudaSuccess && tb) e = cudaMemcpyAsync(base + off_tiles, wl->tiles.data(), tb, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess && rb) e = cudaMemcpyAsync(base + off_runs, wl->runs.data(), rb, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return set_error(CPATTN_CUDA_ERROR, std::string("work-list upload: ") + cudaGetErrorString(e));

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
  a.tiles = reinterpret_cast<const cpattn::QTile*>(base + off_tiles);
  a.runs = reinterpret_cast<const cpattn::KvRun*>(base + off_runs);
  a.n_tiles = (int32_t)wl->tiles.size();
  a.total_pieces = wl->total_kv_tiles;
  a.max_pieces = wl->tiles.empty() ? 0 : wl->tiles.front().n_kv_tiles;  // longest first
  a.o = o;
  a.partial = false;
  a.lse = lse;
  a.lse_ld = plan->T;
  a.ws = reinterpret_cast<cpattn::WsHeader*>(base);
  a.stream = stream;
  std::string err;
  e = bf16 ? cpattn::launch_attn_bf16_tc(a, &err) : cpattn::launch_attn_fp32_simt(a, &err);
  if (e != cudaSuccess) {
    if (!err.empty()) return set_error(CPATTN_INVALID_ARG, err);
    return set_error(CPATTN_CUDA_ERROR, std::string("attention kernel launch: ") + cudaGetErrorString(e));
  }
  return CPATTN_OK;
}

extern "C" cpattn_status_t cpattn_static_sync_status(void* stream_ptr) {
  using cpattn::set_error;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return set_error(CPATTN_CUDA_ERROR, std::string("stream synchronize: ") + cudaGetErrorString(e));
  // The header of the current device's array, copied by symbol into host stack memory.
  cpattn::WsHeader h;
  e = cudaMemcpyFromSymbol(&h, g_cpattn_static_scratch, sizeof(h), 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return set_error(CPATTN_CUDA_ERROR, std::string("reading the static scratch fault word: ") + cudaGetErrorString(e));
  if (h.fault != 0)
    return set_error(CPATTN_DEVICE_FAULT, "kernel fault " + std::to_string(h.fault) + " in block " +
                                              std::to_string(h.info) + " at " + std::to_string(h.detail) +
                                              " (static scratch)");
  return CPATTN_OK;
}
