// bf16 packed varlen attention backward on the 5th-generation tensor cores.
//
// The backward of blockwise ring attention ("Scaling video training with
// parallelism", section 2, Ring Attention: KV blocks travel around the ring
// while each rank works on its own queries): for the KV shard of virtual rank
// k the gradients dK, dV gather contributions from the queries of rank
// (k + t) mod cp at ring step t, and every query collects dQ from every KV
// shard it sees.  With P = exp(s - lse) recomputed from the saved LSE and
// delta = rowsum(dO * O):
//     dV += P^T dO      dP = dO V^T      dS = P (dP - delta)
//     dK += scale dS^T Q                  dQ += scale dS K
//
// A work item is one KV tile (up to 128 keys of one sequence: inside one
// rank's chunk for a ring step, cut from the sequence for a whole call) of
// one KV head.  It walks, for each query head of the group, the query runs
// that see it in ring order, 64 queries at a time; dK and dV stay in TMEM for
// the whole item and are written once, and each piece's dQ leaves through
// fp32 reductions into a global accumulator.  Items run in groups of KV heads
// (see item_of).
//
// Persistent blocks, one per SM (all 512 TMEM columns):
//   TMEM  S^T[2] (2 x 64) | dP^T[2] (2 x 64) | dV (128) | dK (128)
//         dP^T buffer j & 1 holds dP^T_j, then dS^T_j (bf16, first 32
//         columns), then dQ^T_j: Y issues dQ^T_j after dK_j, and one
//         thread's MMAs run in issue order.
// Warp roles (352 threads):
//   warp 0      producer: K and V per item, Q_j and dO_j per piece through a
//               ring of NSTAGE stages (TMA; a stage is refilled once dK_j,
//               its last reader, has run), and the piece's -lse*log2(e) and -scale*delta
//               (plain loads by the 32 lanes) into shared memory.
//   warp 1      TMEM allocator and MMA issuer X (one thread), per piece j:
//                 S^T_j  = K Q_j^T   (M=128 keys, N=64, K=D)        SS
//                 dP^T_j = V dO_j^T  (M=128, N=64, K=D)             SS
//   warp 10     MMA issuer Y (one thread), per piece j:
//                 dV    += P^T_j dO_j (M=128, N=D, K=64)           TS, A = P^T from TMEM
//                 dK    += dS^T_j Q_j (M=128, N=D, K=64)           TS, A = dS^T from TMEM
//                 dQ^T_j = K^T dS^T_j (M=D, N=64, K=128 keys)      SS, both MN-major
//               One thread cannot issue products with both operands in
//               shared memory faster than about one per 96 cycles, well under
//               the tensor pipe's rate; two issuing threads keep twice as many
//               in flight.  X reuses S buffer j & 1 once Y's dV_{j-2} has read
//               P^T_{j-2}, and dP^T buffer j & 1 once the dQ warps have read
//               dQ^T_{j-2}.
//   warps 2-5   one key per thread: P^T from S^T (exp2 with the saved LSE,
//               causal mask from token positions), written back to TMEM as
//               bf16; dS^T from dP^T, written to TMEM (for dK) and to shared
//               memory (the B operand of dQ^T); at the end of the item dK and
//               dV from TMEM to global memory, staged in the warp's own rows of
//               the two dS^T buffers and written by tensor stores.
//   warps 6-9   one head-dim column per thread: read dQ^T_j from TMEM into a
//               [64 queries][D] fp32 tile in shared memory (NDQ buffers); one
//               thread adds the tile to the fp32 dQ accumulator with a TMA
//               reduce-add (performed in L2).  Rows past the piece hold exact
//               zeros (their dS is zero), so the whole 64-row box is added.
//
// Shared-memory operand layouts (SWIZZLE_128B, 1024-byte aligned atoms):
//   K, V:    [128 keys][64 d] boxes.  K-major A of S^T / dP^T; K is also the
//            MN-major A of dQ^T (M = d: 64-wide d blocks one box apart (LBO),
//            8-key groups 1024 B apart (SBO)).
//   Q_j, dO_j: [64 queries][64 d] boxes.  K-major B of S^T / dP^T, MN-major B
//            of dK / dV (N = d).
//   dS^T_j:  [128 keys][64 queries], written by the softmax warps with the
//            same 128-byte swizzle; MN-major B of dQ^T (N = queries).
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

using namespace dev;

namespace {

// Cap on the queries, dO and fp32 dQ of one group of KV heads, about the
// size of L2 (129 MB): larger groups lose the L2 reuse of head-by-head order.
constexpr int64_t kQGroupBytes = 144ll << 20;

struct alignas(64) BwdParams {
  CUtensorMap tm_k, tm_v;   // [rows, Hkv, D], 128-row boxes
  CUtensorMap tm_q, tm_do;  // [rows, H, D], 64-row boxes
  CUtensorMap tm_dq;        // fp32 dQ accumulator [rows, H, D], 64-row boxes, no swizzle
  CUtensorMap tm_dk, tm_dv; // bf16 dK / dV [rows, Hkv, D], 32-row boxes (when kv_tma)
  const QTile* tiles;       // KV tiles (key rows in q_row0 / q_pos0 / q_rows / out_row0)
  const KvRun* runs;        // query runs
  const float* nl2;         // [H, ld]: -lse * log2(e) (-inf for a row with no key)
  const float* nd;          // [H, ld]: -delta
  int64_t ld;
  void* dk;                 // bf16 [*, Hkv, D] stored, or fp32 accumulated (kAccum)
  void* dv;
  const int64_t* out_map;   // optional: output row of a buffer row
  WsHeader* ws;
  int32_t n_tiles, H, Hkv;
  int32_t kv_group;         // KV heads per item group (divides Hkv)
  int32_t kv_tma;           // 1: full 32-row slices of dK / dV leave through tm_dk / tm_dv
  float scale_log2;         // softmax scale * log2(e)
  float scale;              // softmax scale (dS is scaled by it)
};

// NSTAGE: Q/dO ring stages.  Three stages fit beside one dQ staging tile, two
// beside two; the launch picks three for work lists of short items.
template <int D, int NSTAGE>
struct BwdCfg {
  static constexpr int KB = D / 64;
  static constexpr uint32_t KBOX = 128 * 128;  // 128 key rows x 128 bytes
  static constexpr uint32_t QBOX = 64 * 128;   // 64 query rows x 128 bytes
  static constexpr uint32_t KT_BYTES = KB * KBOX;
  static constexpr uint32_t QT_BYTES = KB * QBOX;
  static constexpr uint32_t DS_BYTES = 128 * 128;  // dS^T: 128 keys x 64 queries bf16
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = KT_BYTES;
  static constexpr int NST = NSTAGE;                          // Q/dO ring stages
  static constexpr int NDQ = NSTAGE >= 3 ? 1 : 2;             // dQ staging tiles
  static constexpr uint32_t OFF_Q = 2 * KT_BYTES;             // Q[NST]
  static constexpr uint32_t OFF_DO = OFF_Q + NST * QT_BYTES;  // dO[NST]
  static constexpr uint32_t OFF_DS = OFF_DO + NST * QT_BYTES; // dS^T[2]
  static constexpr uint32_t DQS_BYTES = 64 * D * 4;          // dQ staging tile (fp32)
  static constexpr uint32_t OFF_DQS = OFF_DS + 2 * DS_BYTES;  // [NDQ]
  static constexpr uint32_t OFF_LD = OFF_DQS + NDQ * DQS_BYTES;  // [NST stages][nl2 64 | nd 64] floats
  static constexpr uint32_t OFF_BAR = OFF_LD + NST * 512;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 384;         // 43 mbarriers (344 bytes) below
  static constexpr uint32_t SMEM = OFF_MISC + 64 + 1024;      // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // S^T[2] | dP^T[2] (dP^T_j, then dS^T_j over its first 32 columns, then dQ^T_j) | dV | dK
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384;
};

// Walks the query runs of an item in pieces of up to 64 queries, once per
// query head of the KV head's group.
struct Piece {
  int row0, pos0, len, causal, hq;
};
struct QCursor {
  int r, off, r_begin, r_end, hq;
  __device__ Piece next(const KvRun* runs) {
    Piece pc{0, 0, 0, 0, hq};
    const KvRun run = runs[r];
    pc.row0 = run.kv_row0 + off;
    pc.pos0 = run.kv_pos0 + off;
    pc.len = min(64, run.kv_len - off);
    pc.causal = run.causal;
    off += 64;
    if (off >= run.kv_len) {
      off = 0;
      if (++r >= r_end) {
        r = r_begin;
        ++hq;
      }
    }
    return pc;
  }
};

struct Item {
  int tile_id, g;
};
// Items run in groups of kv_group KV heads; inside a group, KV tile by KV
// tile in the work list's longest-first order, each tile for every KV head of
// the group (the group's queries, dO and dQ stay in L2 while it runs).
__device__ __forceinline__ Item item_of(int i, int n_tiles, int kv_group) {
  const int per_group = n_tiles * kv_group;
  const int grp = i / per_group;
  const int r = i - grp * per_group;
  return Item{r / kv_group, grp * kv_group + r % kv_group};
}

template <int D, bool kAccum, int NSTAGE>
__global__ void __launch_bounds__(352, 1) attn_bwd_tc_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D, NSTAGE>;
  constexpr uint32_t IDESC_ST = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t IDESC_KV = idesc_bf16_f32(128, D, false, true);
  constexpr uint32_t IDESC_DQ = idesc_bf16_f32(D, 64, true, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* qd_full = bars + 2;    // [NST] Q_j and dO_j landed
  uint64_t* qd_empty = bars + 5;   // [NST] dK_j, the last MMA that reads stage j % NST, has run
  uint64_t* ld_full = bars + 8;    // [NST] -lse2 / -scale*delta of piece j in shared memory
  uint64_t* s_full = bars + 11;    // [2]
  uint64_t* p_full = bars + 13;    // [2]
  uint64_t* acc_done = bars + 15;  // the item's last dK / dV MMA has run
  uint64_t* acc_free = bars + 16;  // the epilogue has read dK / dV
  uint64_t* drain = bars + 17;
  uint64_t* drain_y = bars + 18;
  uint64_t* item_full = bars + 19;   // [4]
  uint64_t* item_empty = bars + 23;  // [4]
  uint64_t* stage_full = bars + 27;  // [NDQ] a dQ staging tile is written
  uint64_t* stage_free = bars + 29;  // [NDQ] its previous reduce has read it
  uint64_t* s_free = bars + 31;      // [2] dV_j has read P^T_j: S buffer j & 1 may be overwritten
  uint64_t* dp_full = bars + 33;     // [2] dP^T_j has run
  uint64_t* dq_free = bars + 35;     // [2] the dQ warps have read dQ^T_j: dP^T buffer j & 1 is free
  uint64_t* dq_ready = bars + 37;    // [2] dQ^T_j, piece j's last MMA, has run (its dS^T buffer is free)
  // dS^T_j written to TMEM (dK_j may start) and to shared memory (dQ^T_j may
  // start), one barrier per piece parity: a softmax warp may run a piece
  // ahead of the others, so consecutive pieces cannot share a barrier's phases
  uint64_t* ds_full = bars + 39;       // [2]
  uint64_t* ds_smem_full = bars + 41;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  int* issued = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);     // loads issued: [0] K/V, [1] Q/dO
  int* item_ring = reinterpret_cast<int*>(smem + C::OFF_MISC + 32);  // [4]
  float* ldv = reinterpret_cast<float*>(smem + C::OFF_LD);           // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.H / p.Hkv;
  const int n_items = p.n_tiles * p.Hkv;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int st = 0; st < C::NST; ++st) {
      mbar_init(qd_full + st, 1);
      mbar_init(qd_empty + st, 1);
      mbar_init(ld_full + st, 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ds_full + b, 128);
      mbar_init(ds_smem_full + b, 128);
    }
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 128);
    mbar_init(drain, 1);
    mbar_init(drain_y, 1);
    mbar_init(s_free, 1);
    mbar_init(s_free + 1, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(dp_full + b, 1);
      mbar_init(dq_free + b, 128);
      mbar_init(dq_ready + b, 1);
    }
    for (int r = 0; r < 4; ++r) {
      mbar_init(item_full + r, 1);
      mbar_init(item_empty + r, 258);  // two MMA threads + 128 softmax + 128 dQ threads
    }
    for (int q = 0; q < C::NDQ; ++q) {
      mbar_init(stage_full + q, 128);
      mbar_init(stage_free + q, 1);
    }
    *abort_flag = 0;
    issued[0] = issued[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto take_item = [&](int k, uint32_t where) -> int {
    if (!wait_bounded(item_full + (k & 3), (k >> 2) & 1, abort_flag, p.ws, where)) return -2;
    const int i = item_ring[k & 3];
    mbar_arrive(item_empty + (k & 3));
    return i;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (whole warp)
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
    }
    int g = 0, kc = 0;
    bool ok = true;
    int i = blockIdx.x;
    for (int k = 0; ok; ++k) {
      if (k >= 4 &&
          !__all_sync(0xffffffffu, wait_bounded(item_empty + (k & 3), ((k >> 2) - 1) & 1, abort_flag, p.ws, 1)))
        break;
      if (lane == 0) {
        item_ring[k & 3] = (i < n_items) ? i : -1;
        mbar_arrive(item_full + (k & 3));
      }
      if (i >= n_items) break;
      const Item it = item_of(i, p.n_tiles, p.kv_group);
      const QTile tile = p.tiles[it.tile_id];
      int nxt = 0;
      if (lane == 0) nxt = (int)gridDim.x + (int)atomicAdd(&p.ws->next_item, 1u);
      i = __shfl_sync(0xffffffffu, nxt, 0);
      const int n = tile.n_kv_tiles * G;
      if (n == 0) continue;
      // K and V of this item once the previous item's MMAs are done with them
      if (kc > 0 && !__all_sync(0xffffffffu, wait_bounded(kv_empty, (kc - 1) & 1, abort_flag, p.ws, 2))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::KT_BYTES);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(smem + C::OFF_K + kb * C::KBOX, &p.tm_k, kv_full, kb * 64, it.g, tile.q_row0);
          tma_load_3d(smem + C::OFF_V + kb * C::KBOX, &p.tm_v, kv_full, kb * 64, it.g, tile.q_row0);
        }
        issued[0] = kc + 1;
      }
      ++kc;
      QCursor cur{tile.run_begin, 0, tile.run_begin, tile.run_end, 0};
      for (int t = 0; t < n; ++t, ++g) {
        const Piece pc = cur.next(p.runs);
        const int h = it.g * G + pc.hq;
        const int st = g % C::NST;
        if (g >= C::NST &&
            !__all_sync(0xffffffffu, wait_bounded(qd_empty + st, (g / C::NST - 1) & 1, abort_flag, p.ws, 3))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(qd_full + st, 2 * C::QT_BYTES);
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(smem + C::OFF_Q + st * C::QT_BYTES + kb * C::QBOX, &p.tm_q, qd_full + st, kb * 64, h, pc.row0);
            tma_load_3d(smem + C::OFF_DO + st * C::QT_BYTES + kb * C::QBOX, &p.tm_do, qd_full + st, kb * 64, h,
                        pc.row0);
          }
          issued[1] = g + 1;
        }
        // the piece's -lse*log2(e) and -scale*delta (columns past the piece: -inf and 0, so P = 0 there)
        float* dst = ldv + st * 128;
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          const int c = c0 + lane;
          const bool in = c < pc.len;
          const int64_t src = (int64_t)h * p.ld + pc.row0 + (in ? c : 0);
          dst[c] = in ? p.nl2[src] : -INFINITY;
          dst[64 + c] = in ? p.nd[src] * p.scale : 0.f;
        }
        mbar_arrive(ld_full + st);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer X
    if (lane == 0) {
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      // X^T_g = A B_g^T with A = K or V (K-major), B_g = Q or dO of piece g (K-major)
      auto issue_t = [&](uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * C::KBOX + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * C::QBOX + (kk & 3) * 32;
          umma_bf16_ss(d_tmem, smem_desc_sw128(a_base + aoff, 16, 1024), smem_desc_sw128(b_base + boff, 16, 1024),
                       IDESC_ST, kk > 0 ? 1u : 0u);
        }
      };
      // S^T_j and dP^T_j, the products that read K and V from shared memory.
      // S^T_j reuses the S buffer of piece j - 2 once dV_{j-2} has read its
      // P^T; dP^T_j reuses the dP^T buffer once dK_{j-1} has read its dS^T.
      int g = 0, kc = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int i = take_item(k, 5);
        if (i < 0) break;
        const int n = p.tiles[item_of(i, p.n_tiles, p.kv_group).tile_id].n_kv_tiles * G;
        if (n == 0) continue;
        ok = wait_bounded(kv_full, kc & 1, abort_flag, p.ws, 6);
        if (!ok) break;
        ++kc;
        for (int t = 0; ok && t < n; ++t, ++g) {
          const int b = g & 1, st = g % C::NST;
          ok = wait_bounded(qd_full + st, (g / C::NST) & 1, abort_flag, p.ws, 7);
          if (ok && g >= 2) ok = wait_bounded(s_free + b, ((g >> 1) - 1) & 1, abort_flag, p.ws, 10);
          if (!ok) break;
          tc_fence_after();
          issue_t(tmem + C::TM_S + 64u * b, sK, sQ + st * C::QT_BYTES);
          umma_commit(s_full + b);
          // dP^T buffer b last held dQ^T_{g-2}: the dQ warps must have read it
          if (g >= 2) ok = wait_bounded(dq_free + b, ((g >> 1) - 1) & 1, abort_flag, p.ws, 23);
          if (!ok) break;
          tc_fence_after();
          issue_t(tmem + C::TM_DP + 64u * b, sV, sDO + st * C::QT_BYTES);
          umma_commit(dp_full + b);
        }
      }
      umma_commit(drain);
      drain_wait(drain, 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ P / dS (one key per thread) + epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    const float c2 = p.scale_log2;
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    int g = 0, ac = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int i = take_item(k, 13);
      if (!__all_sync(0xffffffffu, i != -2)) break;
      if (i < 0) break;
      const Item it = item_of(i, p.n_tiles, p.kv_group);
      const QTile tile = p.tiles[it.tile_id];
      const int n = tile.n_kv_tiles * G;
      const bool key_ok = row < tile.q_rows;
      const int kp = tile.q_pos0 + row;
      const int kp_last = tile.q_pos0 + tile.q_rows - 1;
      QCursor cur{tile.run_begin, 0, tile.run_begin, tile.run_end, 0};
      for (int t = 0; t < n; ++t, ++g) {
        const Piece pc = cur.next(p.runs);
        const int b = g & 1;
        const int st = g % C::NST;
        if (!__all_sync(0xffffffffu, wait_bounded(s_full + b, (g >> 1) & 1, abort_flag, p.ws, 14) &&
                                         wait_bounded(ld_full + st, (g / C::NST) & 1, abort_flag, p.ws, 15))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* nl2 = ldv + st * 128;
        const float* nd = nl2 + 64;
        float P[64];
        {
          uint32_t sr[64];
          tmem_ld64_wait(tl + C::TM_S + 64u * b, sr);
          const float2 c2v = make_float2(c2, c2);
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])), c2v,
                                        make_float2(nl2[2 * q], nl2[2 * q + 1]));
            P[2 * q] = ex2_approx(x.x);
            P[2 * q + 1] = ex2_approx(x.y);
          }
        }
        if (!key_ok) {
#pragma unroll
          for (int c = 0; c < 64; ++c) P[c] = 0.f;
        } else if (pc.causal && pc.pos0 < kp_last) {
          const int lim = kp - pc.pos0;  // query column c sees this key iff c >= lim
#pragma unroll
          for (int c = 0; c < 64; ++c) P[c] = (c >= lim) ? P[c] : 0.f;
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) pk[q] = pack_bf16x2(P[2 * q], P[2 * q + 1]);
          tmem_st32(tl + C::TM_S + 64u * b, pk);  // P^T over the first 32 columns of this S buffer
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + b);

        if (!__all_sync(0xffffffffu, wait_bounded(dp_full + b, (g >> 1) & 1, abort_flag, p.ws, 16))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t ds[32];
        {
          uint32_t dr[64];
          tmem_ld64_wait(tl + C::TM_DP + 64u * b, dr);
          // dS = P * (scale * dP - scale * delta), two queries per packed FMA and multiply
          const float2 sc2 = make_float2(p.scale, p.scale);
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const float2 t = __ffma2_rn(make_float2(__uint_as_float(dr[2 * q]), __uint_as_float(dr[2 * q + 1])), sc2,
                                        make_float2(nd[2 * q], nd[2 * q + 1]));
            const float2 a = __fmul2_rn(make_float2(P[2 * q], P[2 * q + 1]), t);
            ds[q] = pack_bf16x2(a.x, a.y);
          }
        }
        tmem_st32(tl + C::TM_DP + 64u * b, ds);  // dS^T (A of dK) over the first 32 columns of dP^T
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_full + b);  // dK_j may start; dQ^T_j waits for the copy below
        // dS^T for dQ^T: this buffer was last read by the dQ^T MMA of piece g - 2
        if (g >= 2 &&
            !__all_sync(0xffffffffu, wait_bounded(dq_ready + b, ((g >> 1) - 1) & 1, abort_flag, p.ws, 17))) {
          ok = false;
          break;
        }
        {
          const uint32_t rbase = sDS + b * C::DS_BYTES + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(rbase + ((c ^ (row & 7)) << 4), ds[4 * c], ds[4 * c + 1], ds[4 * c + 2], ds[4 * c + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(ds_smem_full + b);
      }
      if (!ok) break;

      // epilogue: dK and dV of this KV tile
      if (n > 0) {
        if (!__all_sync(0xffffffffu, wait_bounded(acc_done, ac & 1, abort_flag, p.ws, 18))) break;
        tc_fence_after();
      }
      const int64_t out_row = p.out_map ? p.out_map[tile.out_row0 + (key_ok ? row : 0)]
                                        : (int64_t)tile.out_row0 + row;
      bool acc_read = false;
      if (!kAccum && p.kv_tma && n > 0 && quad * 32 + 32 <= tile.q_rows) {
        // All 32 key rows of this warp are valid: dV, then dK, leave through a
        // tensor store each, staged in the warp's own rows of the two dS^T
        // buffers (64 columns in each), which are free once the item's last
        // dQ^T has run (Y's MMAs complete in issue order) and which no other
        // warp writes.
        if (!__all_sync(0xffffffffu, wait_bounded(dq_ready + ((g - 1) & 1), ((g - 1) >> 1) & 1, abort_flag, p.ws, 20)))
          break;
        uint8_t* stg = smem + C::OFF_DS + quad * 4096;  // + hf * DS_BYTES: the rows in buffer hf
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t tcol = which ? C::TM_DK : C::TM_DV;
          if (which == 1) {
            // dV's stores must have read the slice first
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
          }
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            uint32_t v[64];
            tmem_ld64_wait(tl + tcol + 64u * hf, v);
            if (which == 1 && hf == D / 64 - 1) {
              // dK and dV have been read: the next item's first dV / dK may overwrite them
              tc_fence_before();
              mbar_arrive(acc_free);
              acc_read = true;
            }
            const uint32_t row_addr = smem_u32(stg + hf * C::DS_BYTES) + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)  // 16-byte chunk c of the row, 128-byte swizzle
              st_shared_v4(row_addr + ((c ^ (lane & 7)) << 4),
                           pack_bf16x2(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              tma_store_3d(which ? &p.tm_dk : &p.tm_dv, stg + hf * C::DS_BYTES, 64 * hf, it.g, (int)out_row);
            bulk_commit_group();
          }
        }
        // the next item's dS^T copies may overwrite the slice once the stores have read it
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      } else {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          void* base = which ? p.dk : p.dv;
          const uint32_t tcol = which ? C::TM_DK : C::TM_DV;
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t v[32];
            if (n > 0) {
              tmem_ld32_wait(tl + tcol + 32u * cb, v);
            } else {
#pragma unroll
              for (int q = 0; q < 32; ++q) v[q] = 0u;
            }
            if (!key_ok) continue;
            if (kAccum) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + (out_row * p.Hkv + it.g) * D + 32 * cb);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                float4 a = dst[q];
                a.x += __uint_as_float(v[4 * q]);
                a.y += __uint_as_float(v[4 * q + 1]);
                a.z += __uint_as_float(v[4 * q + 2]);
                a.w += __uint_as_float(v[4 * q + 3]);
                dst[q] = a;
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + (out_row * p.Hkv + it.g) * D +
                                                    32 * cb);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(
                    pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                    pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                    pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                    pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
            }
          }
        }
      }
      if (n > 0) {
        if (!acc_read) {
          tc_fence_before();
          mbar_arrive(acc_free);
        }
        ++ac;
      }
    }
    if (lane == 0) bulk_wait_group_all();  // this warp's tensor stores of dK / dV have completed
  } else if (warp < 10) {
    // ------------------------------------------------------------ dQ (one head-dim column per thread)
    const int quad = warp & 3;
    const int d = quad * 32 + lane;
    const bool leader = (warp == 6 && lane == 0);
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    float* stage = reinterpret_cast<float*>(smem + C::OFF_DQS);
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int i = take_item(k, 19);
      if (!__all_sync(0xffffffffu, i != -2)) break;
      if (i < 0) break;
      const Item it = item_of(i, p.n_tiles, p.kv_group);
      const QTile tile = p.tiles[it.tile_id];
      const int n = tile.n_kv_tiles * G;
      QCursor cur{tile.run_begin, 0, tile.run_begin, tile.run_end, 0};
      for (int t = 0; t < n; ++t, ++g) {
        const Piece pc = cur.next(p.runs);
        const int sb = g & 1;
        // every MMA of piece g, dQ^T_g the last, has run
        if (!__all_sync(0xffffffffu, wait_bounded(dq_ready + (g & 1), (g >> 1) & 1, abort_flag, p.ws, 20))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[64];
        tmem_ld64_wait(tl + C::TM_DP + 64u * sb, v);
        tc_fence_before();
        mbar_arrive(dq_free + sb);
        // staging tile g % NDQ: the reduce of piece g - NDQ must have read it
        const int tq = g % C::NDQ;
        if (leader) {
          bulk_wait_group_read<C::NDQ - 1>();
          mbar_arrive(stage_free + tq);
        }
        if (!__all_sync(0xffffffffu, wait_bounded(stage_free + tq, (g / C::NDQ) & 1, abort_flag, p.ws, 21))) {
          ok = false;
          break;
        }
        float* st = stage + tq * (64 * D);
#pragma unroll
        for (int c = 0; c < 64; ++c) st[c * D + d] = __uint_as_float(v[c]);
        fence_proxy_async_smem();
        mbar_arrive(stage_full + tq);
        if (leader) {
          if (!wait_bounded(stage_full + tq, (g / C::NDQ) & 1, abort_flag, p.ws, 22)) {
            ok = false;
          } else {
            tma_reduce_add_3d(&p.tm_dq, st, 0, it.g * G + pc.hq, pc.row0);
            bulk_commit_group();
          }
        }
        if (!__all_sync(0xffffffffu, ok)) break;
      }
    }
    // every reduce has finished before the block exits
    if (leader) bulk_wait_group_all();
  } else {
    // ------------------------------------------------------------ MMA issuer Y
    // dV_j, dK_j and dQ^T_j: the products that read P^T_j and dS^T_j.  A second
    // issuing thread, so that the shared-memory operand products of the two
    // threads are in flight together.
    if (lane == 0) {
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS);
      int g = 0, ac = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int i = take_item(k, 24);
        if (i < 0) break;
        const int n = p.tiles[item_of(i, p.n_tiles, p.kv_group).tile_id].n_kv_tiles * G;
        if (n == 0) continue;
        for (int t = 0; ok && t < n; ++t, ++g) {
          const int b = g & 1;
          ok = wait_bounded(p_full + b, (g >> 1) & 1, abort_flag, p.ws, 8);
          // the item's first dV / dK overwrite the accumulators: the previous epilogue must have read them
          if (ok && t == 0 && ac > 0) ok = wait_bounded(acc_free, (ac - 1) & 1, abort_flag, p.ws, 9);
          if (!ok) break;
          tc_fence_after();
          const int st = g % C::NST;
          const uint32_t qb = sQ + st * C::QT_BYTES, dob = sDO + st * C::QT_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dV += P^T dO: 16 queries per MMA
            umma_bf16_ts(tmem + C::TM_DV, tmem + C::TM_S + 64u * b + 8 * kk,
                         smem_desc_sw128(dob + kk * 2048, C::QBOX, 1024), IDESC_KV, (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(s_free + b);
          ok = wait_bounded(ds_full + b, (g >> 1) & 1, abort_flag, p.ws, 11);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // dK += dS^T Q
            umma_bf16_ts(tmem + C::TM_DK, tmem + C::TM_DP + 64u * b + 8 * kk, smem_desc_sw128(qb + kk * 2048, C::QBOX, 1024),
                         IDESC_KV, (t > 0 || kk > 0) ? 1u : 0u);
          umma_commit(qd_empty + st);  // stage st (Q_g, dO_g) may be refilled
          ok = wait_bounded(ds_smem_full + b, (g >> 1) & 1, abort_flag, p.ws, 25);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dsb = sDS + b * C::DS_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ^T = K^T dS^T: 16 keys per MMA
            umma_bf16_ss(tmem + C::TM_DP + 64u * b, smem_desc_sw128(sK + kk * 2048, C::KBOX, 1024),
                         smem_desc_sw128(dsb + kk * 2048, C::DS_BYTES, 1024), IDESC_DQ, kk > 0 ? 1u : 0u);
          umma_commit(dq_ready + b);  // the dQ warps may read dQ^T_g; dS^T buffer b is free
          if (t == n - 1) {
            umma_commit(acc_done);
            umma_commit(kv_empty);
          }
        }
        ++ac;
      }
      umma_commit(drain_y);
      drain_wait(drain_y, 0);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      if (issued[0]) drain_wait(kv_full, (issued[0] - 1) & 1);
      for (int gg = max(0, issued[1] - C::NST); gg < issued[1]; ++gg)
        drain_wait(qd_full + gg % C::NST, (gg / C::NST) & 1);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// delta = rowsum(dO * O), -lse * log2(e) and (optionally) a zeroed dQ
// accumulator row.  A group of D*sizeof(T)/16 lanes (16-byte loads) per
// (buffer row, head); rows of O, dO and LSE are read at in_map[row] when a map
// is given (buffers of gathered shards).
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                      const float* __restrict__ lse, int64_t lse_ld,
                                                      const int64_t* __restrict__ in_map, int64_t rows, int H,
                                                      float* __restrict__ nl2, float* __restrict__ nd,
                                                      float* __restrict__ dq_zero) {
  constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte load
  constexpr int kLanes = D / kPer;      // lanes per (row, head): 8 or 16 (bf16), 16 or 32 (fp32)
  const int64_t gid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kLanes;
  const int sub = threadIdx.x % kLanes;
  const bool active = gid < rows * H;
  const int64_t row = active ? gid / H : 0;
  const int h = active ? (int)(gid % H) : 0;
  const int64_t src = active ? (in_map ? in_map[row] : row) : 0;
  float acc = 0.f;
  if (active) {
    const uint4 a = reinterpret_cast<const uint4*>(o + (src * H + h) * D)[sub];
    const uint4 b = reinterpret_cast<const uint4*>(dout + (src * H + h) * D)[sub];
    const T* av = reinterpret_cast<const T*>(&a);
    const T* bv = reinterpret_cast<const T*>(&b);
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc += (float)av[e] * (float)bv[e];
  }
#pragma unroll
  for (int s = kLanes / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (!active) return;
  if (sub == 0) {
    const float l = lse[(int64_t)h * lse_ld + src];
    nl2[(int64_t)h * rows + row] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
    nd[(int64_t)h * rows + row] = -acc;
  }
  if (dq_zero) {
    float4* z = reinterpret_cast<float4*>(dq_zero + (row * H + h) * D);
    for (int c = sub; c < D / 4; c += kLanes) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// From the fp32 dQ accumulator (buffer rows) to the output: row r goes to
// map[r] (or r); kAdd adds to a fp32 output, else the value is stored in the
// output dtype.  Four elements per thread.
template <typename T, bool kAdd>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float4* __restrict__ acc, T* __restrict__ out,
                                                       int64_t n4, int64_t row4, const int64_t* __restrict__ map) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const int64_t row = i / row4, c = i - row * row4;
  const int64_t dst = (map ? map[row] : row) * row4 + c;
  const float4 a = acc[i];
  if constexpr (kAdd) {
    float4* o = reinterpret_cast<float4*>(out) + dst;
    float4 x = *o;
    x.x += a.x;
    x.y += a.y;
    x.z += a.z;
    x.w += a.w;
    *o = x;
  } else if constexpr (sizeof(T) == 2) {
    reinterpret_cast<uint2*>(out)[dst] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  } else {
    reinterpret_cast<float4*>(out)[dst] = a;
  }
}

template <int D, bool kAccum, int NSTAGE>
cudaError_t launch_bwd_tc(const BwdParams& p, int n_blocks, cudaStream_t stream) {
  auto kern = attn_bwd_tc_kernel<D, kAccum, NSTAGE>;
  const uint32_t smem = BwdCfg<D, NSTAGE>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<n_blocks, 352, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

template <typename T, int D>
static void pre_launch(const BwdArgs& a) {
  constexpr int kLanes = D / (16 / sizeof(T));
  const int64_t threads = a.rows_total * a.H * kLanes;
  bwd_pre_kernel<T, D><<<(unsigned)((threads + 255) / 256), 256, 0, a.stream>>>(
      static_cast<const T*>(a.o), static_cast<const T*>(a.dout), a.lse, a.lse_ld, a.in_map, a.rows_total, a.H,
      a.nl2, a.nd, a.zero_dq ? a.dq_acc : nullptr);
}

cudaError_t launch_bwd_pre(const BwdArgs& a) {
  if (a.rows_total * a.H == 0) return cudaSuccess;
  if (a.bf16)
    a.D == 128 ? pre_launch<__nv_bfloat16, 128>(a) : pre_launch<__nv_bfloat16, 64>(a);
  else
    a.D == 128 ? pre_launch<float, 128>(a) : pre_launch<float, 64>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(const float* dq_acc, void* out, bool out_bf16, bool add, int64_t rows,
                            int64_t row_elems, const int64_t* map, cudaStream_t stream) {
  const int64_t n4 = rows * row_elems / 4, row4 = row_elems / 4;
  if (n4 == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((n4 + 255) / 256);
  const float4* acc = reinterpret_cast<const float4*>(dq_acc);
  if (add)
    bwd_post_kernel<float, true><<<blocks, 256, 0, stream>>>(acc, static_cast<float*>(out), n4, row4, map);
  else if (out_bf16)
    bwd_post_kernel<__nv_bfloat16, false><<<blocks, 256, 0, stream>>>(acc, static_cast<__nv_bfloat16*>(out), n4,
                                                                      row4, map);
  else
    bwd_post_kernel<float, false><<<blocks, 256, 0, stream>>>(acc, static_cast<float*>(out), n4, row4, map);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_bf16_tc(const BwdArgs& a, std::string* err) {
  if (a.D != 128) {
    *err = "the bf16 backward supports D = 128";
    return cudaErrorInvalidValue;
  }
  BwdParams p;
  memset(&p, 0, sizeof(p));
  if (!make_tensor_map_bf16(&p.tm_k, a.k, a.rows_total, a.Hkv, a.D, 128, err) ||
      !make_tensor_map_bf16(&p.tm_v, a.v, a.rows_total, a.Hkv, a.D, 128, err) ||
      !make_tensor_map_bf16(&p.tm_q, a.q, a.rows_total, a.H, a.D, 64, err) ||
      !make_tensor_map_bf16(&p.tm_do, a.dout_rows, a.rows_total, a.H, a.D, 64, err) ||
      !make_tensor_map_f32(&p.tm_dq, a.dq_acc, a.rows_total, a.H, a.D, 64, err))
    return cudaErrorInvalidValue;
  if (!a.accumulate && !a.out_map) {
    // bf16 gradients at contiguous rows: full 32-row slices leave by tensor stores
    if (!make_tensor_map_bf16(&p.tm_dk, a.dk, a.rows_total, a.Hkv, a.D, 32, err) ||
        !make_tensor_map_bf16(&p.tm_dv, a.dv, a.rows_total, a.Hkv, a.D, 32, err))
      return cudaErrorInvalidValue;
    p.kv_tma = 1;
  }
  p.tiles = a.tiles;
  p.runs = a.runs;
  p.nl2 = a.nl2;
  p.nd = a.nd;
  p.ld = a.rows_total;
  p.dk = a.dk;
  p.dv = a.dv;
  p.out_map = a.out_map;
  p.ws = a.ws;
  p.n_tiles = a.n_tiles;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t items = (int64_t)a.n_tiles * a.Hkv;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffff) {
    *err = "too many KV tiles";
    return cudaErrorInvalidValue;
  }
  const int64_t blocks = std::min<int64_t>(items, (int64_t)num_sms());
  // Item groups: the smallest divisor of Hkv whose work per block is at least
  // 1.25 times the longest item, so that the last group's longest items do
  // not run alone at the end, as long as the group's Q, dO and fp32 dQ fit
  // about one L2; past that, the largest divisor that fits.
  p.kv_group = 1;
  const int64_t q_side_bytes = (int64_t)(a.H / a.Hkv) * a.rows_total * a.D * (2 + 2 + 4);
  for (int d = 1; d <= a.Hkv; ++d) {
    if (a.Hkv % d != 0) continue;
    if (d > 1 && d * q_side_bytes > kQGroupBytes) break;
    p.kv_group = d;
    if (4 * (int64_t)d * a.total_pieces >= 5 * (int64_t)a.max_pieces * blocks) break;
  }
  // Short items (the micro-batch's 128-key tiles meet about 20 query pieces
  // each) refill the Q/dO ring at every item start, where a third stage pays;
  // on long items two stages with two dQ staging tiles measured faster.
  if (a.total_pieces < 64 * (int64_t)a.n_tiles)
    return a.accumulate ? launch_bwd_tc<128, true, 3>(p, (int)blocks, a.stream)
                        : launch_bwd_tc<128, false, 3>(p, (int)blocks, a.stream);
  return a.accumulate ? launch_bwd_tc<128, true, 2>(p, (int)blocks, a.stream)
                      : launch_bwd_tc<128, false, 2>(p, (int)blocks, a.stream);
}

}  // namespace cpattn
