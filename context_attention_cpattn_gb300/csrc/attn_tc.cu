// bf16 packed varlen attention forward on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, Q/K/V tiles staged by TMA).
//
// A work item is one 128-row query tile of one head.  It walks the tile's KV
// runs in ring order - at ring step t the queries of virtual rank r see the
// KV shard of rank (r - t) mod cp ("Scaling video training with parallelism",
// section 2, Ring Attention) - in 64-key tiles, and merges every tile's
// partial into the running result by exact log-sum-exp rescaling, so each
// ring step's partial (O_t, lse_t) is folded in as soon as it is produced and
// never leaves the SM.
//
// Persistent blocks, two per SM (113 KB of shared memory, 16 KB of it the
// epilogue's staging area, and 256 TMEM columns each).  The producer warp
// hands out work items (the first by block index, the rest from an atomic
// counter) through a ring of shared-memory slots.  Items run in groups of KV
// heads (see item_of), tile by tile longest first inside a group.
//
// Warp roles (224 threads):
//   warp 0      TMA producer: Q per item, then K and V through two-deep
//               rings in the order the MMAs read them (K_0, K_1, V_0, K_2,
//               V_1, ...); K_j is refilled once S_j has read it, V_j once
//               PV_j has.
//   warp 1      TMEM allocator and S issuer (one thread).  TMEM holds two S
//               buffers of 64 columns and O (128 columns).
//                 S_j  = Q K_j^T  (M=128, N=64, K=D)   A, B from shared memory
//               S_j goes into buffer j & 1 once PV_{j-2} has read the P that
//               buffer held.
//   warp 2      PV issuer (one thread):
//                 O   += P_j V_j  (M=128, N=D,  K=64)  A = P_j from TMEM, B = V_j
//               A tcgen05.mma costs its issuing thread about a hundred cycles
//               whatever its shape, so the two products of a tile issue from
//               two threads, ordered by mbarriers (S_j after PV_{j-2}, PV_j
//               after the softmax of tile j), not by one thread's issue order.
//   warps 3-6   softmax and epilogue, one query row per thread: read S_j from
//               TMEM, apply the causal / run-end mask from token positions,
//               update the running max and sum, write P (bf16 pairs) back over
//               the first 32 columns of S_j's buffer, and rescale O when the
//               running max grows by more than 2^8 (otherwise the stale max is
//               kept: O and the sum share it, so the final O/l is exact).  A
//               rescale first waits for PV_{j-1}.  After an item's last PV they
//               read O, release it for the next item's first PV, and write O/l
//               and the LSE at the output rows: a warp whose 32 rows are all
//               valid (bf16 final outputs at contiguous rows) stages them 64
//               columns at a time in shared memory and writes them with one
//               tensor store, the others store row by row.
//
// Shared-memory operand layouts (1024-byte aligned, SWIZZLE_128B):
//   Q:    [128 rows][64 columns] boxes, K-major.
//   K_j:  [64 keys][64 columns] boxes, K-major (the B operand of S = Q K^T).
//   V_j:  [64 keys][64 d] boxes; as the B operand of P.V (N = d, K = keys)
//         this is MN-major: 8-key groups 1024 B apart (SBO), 64-wide d blocks
//         one box apart (LBO).
// Items of one KV head are consecutive (all its query heads, query tiles
// longest-first), so the KV rows the resident blocks stream stay in L2.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.hpp"

namespace cpattn {

using namespace dev;

// Cap on the keys and values of one group of KV heads, about the size of L2
// (129 MB): larger groups lose the L2 reuse of head-by-head order.
constexpr int64_t kKvGroupBytes = 144ll << 20;

struct alignas(64) TcParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;   // bf16 O [rows, H, D], 64 columns x 1 head x 32 rows boxes (when o_tma)
  const QTile* tiles;
  const KvRun* runs;
  void* o;
  float* lse;
  const int64_t* out_map;
  WsHeader* ws;
  int64_t lse_ld;
  int32_t n_tiles;
  int32_t H, Hkv;
  int32_t kv_group;   // KV heads per item group (divides Hkv)
  int32_t o_tma;      // 1: full 32-row slices of O leave through tm_o
  float scale;        // softmax scale (natural-log domain)
  float scale_log2;   // scale * log2(e)
  float thresh_raw;   // 8 / scale_log2: raw-score growth that forces a rescale
};

template <int D>
struct TcCfg {
  static constexpr int KB = D / 64;                   // 64-column boxes per row
  static constexpr uint32_t QBOX = 128 * 128;         // 128 rows x 128 bytes
  static constexpr uint32_t KVBOX = 64 * 128;         // 64 rows x 128 bytes
  static constexpr uint32_t Q_BYTES = KB * QBOX;
  static constexpr uint32_t KV_BYTES = KB * KVBOX;    // one 64-key K or V tile
  static constexpr uint32_t OFF_K = Q_BYTES;          // K[2]
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;  // V[2]
  static constexpr uint32_t OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 256;  // 29 mbarriers (232 bytes) fit below
  // O staging for the epilogue's tensor stores: per softmax warp 32 rows x 64
  // columns of bf16 (128-byte swizzled rows), at the next 1024-byte boundary
  static constexpr uint32_t OFF_STG = (OFF_MISC + 64 + 1023) / 1024 * 1024;
  static constexpr uint32_t STG_WARP = 32 * 128;
  // No alignment slack: where the dynamic shared memory does not start on a
  // 1024-byte boundary, the layout shifts up by the padding, the staging area
  // no longer fits and the epilogue stores O row by row instead.
  static constexpr uint32_t SMEM = OFF_STG + 4 * STG_WARP;
  static constexpr uint32_t TMEM_COLS = 256;              // S0 | S1 | O
  static constexpr uint32_t TM_S = 0, TM_O = 128;         // S buffer b at TM_S + 64 b
};

// Walks the KV runs of a q tile in tiles of up to 64 keys.
struct Piece {
  int row0, pos0, len, causal;
};
struct PieceCursor {
  int r, off, r_end;
  __device__ Piece next(const KvRun* runs) {
    Piece pc{0, 0, 0, 0};
    if (r >= r_end) return pc;
    const KvRun run = runs[r];
    pc.row0 = run.kv_row0 + off;
    pc.pos0 = run.kv_pos0 + off;
    pc.len = min(64, run.kv_len - off);
    pc.causal = run.causal;
    off += 64;
    if (off >= run.kv_len) {
      ++r;
      off = 0;
    }
    return pc;
  }
};

// Work item i -> (KV head g, query tile, query head inside the group): the
// items of one KV head are consecutive, query tiles longest-first.
struct Item {
  int tile_id, h, g;
};
// Items run in groups of kv_group KV heads; inside a group, tile by tile in
// the work list's longest-first order, each tile for every query head of the
// group.  A group's keys and values stay in L2 while its tiles run, and the
// last group ends on its shortest tiles.
__device__ __forceinline__ Item item_of(int i, int n_tiles, int G, int kv_group) {
  Item it;
  const int span = kv_group * G;  // query heads per group
  const int per_group = n_tiles * span;
  const int grp = i / per_group;
  const int r = i - grp * per_group;
  it.tile_id = r / span;
  const int w = r - it.tile_id * span;
  it.g = grp * kv_group + w / G;
  it.h = it.g * G + w % G;
  return it;
}

template <int D, bool kPartial>
__global__ void __launch_bounds__(224, 2) attn_fwd_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<D>;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem_pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + smem_pad;
  static_assert(C::OFF_MISC + 64 + 1023 <= C::SMEM, "the layout without staging must fit any padding");
  const bool staged = p.o_tma && smem_pad == 0;  // the staging area lies inside the allocation

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;     // [2]
  uint64_t* s_done = bars + 4;     // [2] S_j has run: K_j's buffer is free, the softmax may read S_j
  uint64_t* v_full = bars + 6;     // [2]
  uint64_t* pv_done = bars + 8;    // [2] PV_j has run: V_j's buffer and P_j's S buffer are free, O holds it
  uint64_t* p_full = bars + 12;    // [2]
  uint64_t* o_final = bars + 15;   // after an item's last PV
  uint64_t* o_free = bars + 16;    // the epilogue has read O
  uint64_t* drain = bars + 17;     // the S issuer's MMAs have landed
  uint64_t* item_full = bars + 18;   // [4] ring of work items handed from the producer
  uint64_t* item_empty = bars + 22;  // [4]
  uint64_t* drain2 = bars + 28;      // the PV issuer's MMAs have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  int* issued = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);     // loads issued: [0] K, [1] V, [2] Q
  int* item_ring = reinterpret_cast<int*>(smem + C::OFF_MISC + 32);  // [4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.H / p.Hkv;
  const int n_items = p.n_tiles * p.H;
  // every bounded wait gives up after 4 s, or after the workspace's shorter
  // limit when a fault-path test set one
  const uint64_t wait_ns = p.ws->wait_limit_us ? (uint64_t)p.ws->wait_limit_us * 1000ull : kWaitLimitNs;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(k_full + b, 1);
      mbar_init(s_done + b, 1);
      mbar_init(v_full + b, 1);
      mbar_init(pv_done + b, 1);
      mbar_init(p_full + b, 128);
    }
    mbar_init(o_final, 1);
    mbar_init(o_free, 128);
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    for (int r = 0; r < 4; ++r) {
      mbar_init(item_full + r, 1);
      mbar_init(item_empty + r, 130);  // the two MMA threads and the 128 softmax threads
    }
    *abort_flag = 0;
    issued[0] = issued[1] = issued[2] = 0;
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

  // Items reach the MMA and softmax warps through a 4-deep ring.  KV tiles are
  // counted across items (g), so double-buffered barriers keep alternating
  // phases from one item to the next: buffer g & 1, phase parity (g >> 1) & 1.
  auto take_item = [&](int k, uint32_t where) -> int {  // consumers: item k of this block, or -1
    if (!wait_bounded(item_full + (k & 3), (k >> 2) & 1, abort_flag, p.ws, where, wait_ns)) return -2;
    const int i = item_ring[k & 3];
    mbar_arrive(item_empty + (k & 3));
    return i;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      // fault-path test support: block 0 never loads its first V tile, so the
      // PV issuer's bounded wait for it runs out
      const bool withhold_v0 = (blockIdx.x == 0) && (p.ws->withhold == 1u);
      int g = 0, qc = 0;
      bool ok = true;
      int i = blockIdx.x;
      for (int k = 0; ok; ++k) {
        if (k >= 4 && !wait_bounded(item_empty + (k & 3), ((k >> 2) - 1) & 1, abort_flag, p.ws, 1, wait_ns)) break;
        item_ring[k & 3] = (i < n_items) ? i : -1;
        mbar_arrive(item_full + (k & 3));
        if (i >= n_items) break;
        const Item it = item_of(i, p.n_tiles, G, p.kv_group);
        const QTile tile = p.tiles[it.tile_id];
        i = (int)gridDim.x + (int)atomicAdd(&p.ws->next_item, 1u);
        if (tile.n_kv_tiles == 0) continue;
        // Q of this item once every S MMA of the previous item has read its Q
        if (qc > 0 && !wait_bounded(q_empty, (qc - 1) & 1, abort_flag, p.ws, 2, wait_ns)) break;
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(smem + kb * C::QBOX, &p.tm_q, q_full, kb * 64, it.h, tile.q_row0);
        issued[2] = ++qc;
        // K_{j+1} goes before V_j, the order the MMAs consume them in (S_{j+1}
        // is issued before PV_j); K_{j+1}'s buffer is free once S_{j-1} has
        // run, which precedes PV_{j-2}, the MMA that frees V_j's buffer.
        PieceCursor c{tile.run_begin, 0, tile.run_end};
        auto load_k = [&](int gk, int row) -> bool {
          const int b = gk & 1;
          if (gk >= 2 && !wait_bounded(s_done + b, ((gk >> 1) - 1) & 1, abort_flag, p.ws, 3, wait_ns)) return false;
          mbar_arrive_expect_tx(k_full + b, C::KV_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(smem + C::OFF_K + b * C::KV_BYTES + kb * C::KVBOX, &p.tm_k, k_full + b, kb * 64, it.g, row);
          issued[0] = gk + 1;
          return true;
        };
        int row_next = c.next(p.runs).row0;
        if (!load_k(g, row_next)) break;
        for (int j = 0; j < tile.n_kv_tiles; ++j, ++g) {
          const int row = row_next;
          const int b = g & 1;
          if (j + 1 < tile.n_kv_tiles) {
            row_next = c.next(p.runs).row0;
            if (!load_k(g + 1, row_next)) { ok = false; break; }
          }
          if (g >= 2 && !wait_bounded(pv_done + b, ((g >> 1) - 1) & 1, abort_flag, p.ws, 4, wait_ns)) { ok = false; break; }
          if (withhold_v0 && g == 0) continue;
          mbar_arrive_expect_tx(v_full + b, C::KV_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(smem + C::OFF_V + b * C::KV_BYTES + kb * C::KVBOX, &p.tm_v, v_full + b, kb * 64, it.g, row);
          issued[1] = g + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      const uint32_t sQ = smem_u32(smem), sK = smem_u32(smem + C::OFF_K);
      int g = 0, qc = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int i = take_item(k, 5);
        if (i < 0) break;
        const int n_kv = p.tiles[item_of(i, p.n_tiles, G, p.kv_group).tile_id].n_kv_tiles;
        if (n_kv == 0) continue;
        if (!wait_bounded(q_full, qc & 1, abort_flag, p.ws, 6, wait_ns)) break;
        ++qc;
        for (int j = 0; j < n_kv; ++j, ++g) {
          const int b = g & 1;
          // S_g overwrites the P that PV_{g-2} read
          ok = wait_bounded(k_full + b, (g >> 1) & 1, abort_flag, p.ws, 7, wait_ns) &&
               (g < 2 || wait_bounded(pv_done + b, ((g >> 1) - 1) & 1, abort_flag, p.ws, 11, wait_ns));
          if (!ok) break;
          tc_fence_after();
          const uint32_t kbase = sK + b * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * C::QBOX + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * C::KVBOX + (kk & 3) * 32;
            umma_bf16_ss(tmem + C::TM_S + 64u * b, smem_desc_sw128(sQ + qoff, 16, 1024),
                         smem_desc_sw128(kbase + koff, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
          }
          if (j == n_kv - 1) umma_commit(q_empty);
          umma_commit(s_done + b);
        }
      }
      // every commit above has landed before the block can exit
      umma_commit(drain);
      drain_wait(drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      int g = 0, oc = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int i = take_item(k, 19);
        if (i < 0) break;
        const int n_kv = p.tiles[item_of(i, p.n_tiles, G, p.kv_group).tile_id].n_kv_tiles;
        if (n_kv == 0) continue;
        for (int j = 0; j < n_kv; ++j, ++g) {
          const int b = g & 1;
          ok = wait_bounded(p_full + b, (g >> 1) & 1, abort_flag, p.ws, 8, wait_ns) &&
               wait_bounded(v_full + b, (g >> 1) & 1, abort_flag, p.ws, 9, wait_ns);
          // the first PV of an item overwrites O: the previous item's epilogue must have read it
          if (ok && j == 0 && oc > 0) ok = wait_bounded(o_free, (oc - 1) & 1, abort_flag, p.ws, 10, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vbase = sV + b * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 keys per MMA: P columns 8kk.., V rows 16kk..
            umma_bf16_ts(tmem + C::TM_O, tmem + C::TM_S + 64u * b + 8 * kk,
                         smem_desc_sw128(vbase + kk * 2048, C::KVBOX, 1024), IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(pv_done + b);
          if (j == n_kv - 1) umma_commit(o_final);
        }
        ++oc;
      }
      umma_commit(drain2);
      drain_wait(drain2, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax and epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    const float c2 = p.scale_log2;
    int g = 0, oc = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int i = take_item(k, 12);
      if (!__all_sync(0xffffffffu, i != -2)) break;
      if (i < 0) break;
      const Item it = item_of(i, p.n_tiles, G, p.kv_group);
      const QTile tile = p.tiles[it.tile_id];
      const int n_kv = tile.n_kv_tiles;
      const int q_pos = tile.q_pos0 + row;
      const int q_pos0 = tile.q_pos0;
      float m_ref = -INFINITY, l = 0.f;
      PieceCursor cur{tile.run_begin, 0, tile.run_end};
      for (int j = 0; j < n_kv; ++j, ++g) {
        const Piece pc = cur.next(p.runs);
        const bool tile_mask = (pc.len < 64) || (pc.causal && pc.pos0 + 63 > q_pos0);
        const int b = g & 1;

        if (!__all_sync(0xffffffffu, wait_bounded(s_done + b, (g >> 1) & 1, abort_flag, p.ws, 13, wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64_wait(tl + C::TM_S + 64u * b, sr);
        float s[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c]);
        if (tile_mask) {
          int lim = pc.len;
          if (pc.causal) lim = min(lim, q_pos - pc.pos0 + 1);
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        }
        // row max: four chains of three-input max
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          m0 = fmax3(m0, s[c], s[c + 1]);
          m1 = fmax3(m1, s[c + 2], s[c + 3]);
          m2 = fmax3(m2, s[c + 4], s[c + 5]);
          m3 = fmax3(m3, s[c + 6], s[c + 7]);
        }
        const float mx = fmax3(m0, m1, fmaxf(m2, m3));

        float alpha = 1.f;
        bool scale_o = false;
        if (mx > m_ref + p.thresh_raw) {
          alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx((m_ref - mx) * c2);
          scale_o = (j > 0) && (m_ref != -INFINITY);
          m_ref = mx;
          l *= alpha;
        }
        const float mc = (m_ref == -INFINITY) ? 0.f : m_ref * c2;
        // exponents two at a time on the packed FP32 pipe: x = s*c2 - mc
        const float2 c2v = make_float2(c2, c2), nmc = make_float2(-mc, -mc);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const float2 x = __ffma2_rn(make_float2(s[2 * q], s[2 * q + 1]), c2v, nmc);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (q & 1)
            acc1 = __fadd2_rn(acc1, e);
          else
            acc0 = __fadd2_rn(acc0, e);
          pk[q] = pack_bf16x2(e.x, e.y);
        }
        l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
        tmem_st32(tl + C::TM_S + 64u * b, pk);  // P over the first 32 columns of this S buffer
        if (__any_sync(0xffffffffu, scale_o)) {
          // O may only be rescaled once PV_{g-1} (still in flight) has landed
          if (!__all_sync(0xffffffffu,
                          wait_bounded(pv_done + ((g - 1) & 1), ((g - 1) >> 1) & 1, abort_flag, p.ws, 14, wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float a = scale_o ? alpha : 1.f;
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t o[32];
            tmem_ld32_wait(tl + C::TM_O + 32u * cb, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * a);
            tmem_st32(tl + C::TM_O + 32u * cb, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + b);
      }
      if (!ok) break;
      // ---- epilogue of the item: O/l and the LSE at the output rows
      if (n_kv > 0) {
        if (!__all_sync(0xffffffffu, wait_bounded(o_final, oc & 1, abort_flag, p.ws, 15, wait_ns))) break;
        tc_fence_after();
      }
      const bool valid_row = row < tile.q_rows;
      const bool has = l > 0.f;
      const float inv_l = has ? 1.f / l : 0.f;
      const int64_t out_row = p.out_map ? p.out_map[tile.out_row0 + (valid_row ? row : 0)]
                                        : (int64_t)tile.out_row0 + row;
      if (!kPartial && staged && n_kv > 0 && quad * 32 + 32 <= tile.q_rows) {
        // All 32 rows of this warp are valid: O leaves 64 columns at a time
        // through the warp's staging slice and one tensor store, which writes
        // whole lines instead of 16 bytes of 32 rows per store instruction.
        uint8_t* stg = smem + C::OFF_STG + quad * C::STG_WARP;
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          uint32_t pk[32];  // 64 columns of this row as bf16 pairs
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32_wait(tl + C::TM_O + 64u * hf + 32u * cc, o);
            if (hf == D / 64 - 1 && cc == 1) {
              // O has been read: the next item's first PV may overwrite it
              tc_fence_before();
              mbar_arrive(o_free);
            }
#pragma unroll
            for (int q = 0; q < 16; ++q)
              pk[16 * cc + q] = pack_bf16x2(has ? __uint_as_float(o[2 * q]) * inv_l : 0.f,
                                            has ? __uint_as_float(o[2 * q + 1]) * inv_l : 0.f);
          }
          // the slice is free once the previous tensor store has read it
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          const uint32_t row_addr = smem_u32(stg) + lane * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)  // 16-byte chunk c of the row, 128-byte swizzle
            st_shared_v4(row_addr + ((c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&p.tm_o, stg, 64 * hf, it.h, (int)out_row);
            bulk_commit_group();
          }
        }
      } else {
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          if (n_kv > 0) {
            tmem_ld32_wait(tl + C::TM_O + 32u * cb, o);
            if (cb == D / 32 - 1) {
              // O has been read: the next item's first PV may overwrite it
              tc_fence_before();
              mbar_arrive(o_free);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = 0u;
          }
          if (valid_row) {
            float v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = has ? __uint_as_float(o[q]) * inv_l : 0.f;
            if (kPartial) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + (out_row * p.H + it.h) * D + 32 * cb);
#pragma unroll
              for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              uint4* dst =
                  reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + (out_row * p.H + it.h) * D + 32 * cb);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                    pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
            }
          }
        }
      }
      if (valid_row) p.lse[(int64_t)it.h * p.lse_ld + out_row] = has ? m_ref * p.scale + logf(l) : -INFINITY;
      if (n_kv > 0) ++oc;
    }
    if (lane == 0) bulk_wait_group_all();  // this warp's tensor stores of O have completed
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Let copies and MMAs already in flight land before the block exits.
    if (warp == 0 && lane == 0) {
      if (issued[2]) drain_wait(q_full, (issued[2] - 1) & 1);
      for (int gg = max(0, issued[0] - 2); gg < issued[0]; ++gg) drain_wait(k_full + (gg & 1), (gg >> 1) & 1);
      for (int gg = max(0, issued[1] - 2); gg < issued[1]; ++gg) drain_wait(v_full + (gg & 1), (gg >> 1) & 1);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

template <int D, bool kPartial>
static cudaError_t launch_tc(const TcParams& p, int n_blocks, cudaStream_t stream) {
  auto kern = attn_fwd_tc_kernel<D, kPartial>;
  const uint32_t smem = TcCfg<D>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // two blocks per SM take the whole shared-memory carve-out
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  kern<<<n_blocks, 224, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bf16_tc(const AttnArgs& a, std::string* err) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  if (!make_tensor_map_bf16(&p.tm_q, a.q, a.q_rows_total, a.H, a.D, 128, err) ||
      !make_tensor_map_bf16(&p.tm_k, a.k, a.kv_rows_total, a.Hkv, a.D, 64, err) ||
      !make_tensor_map_bf16(&p.tm_v, a.v, a.kv_rows_total, a.Hkv, a.D, 64, err))
    return cudaErrorInvalidValue;
  if (!a.partial && !a.out_map) {
    // final outputs at contiguous rows: full 32-row slices leave by tensor stores
    if (!make_tensor_map_bf16(&p.tm_o, a.o, a.q_rows_total, a.H, a.D, 32, err)) return cudaErrorInvalidValue;
    p.o_tma = 1;
  }
  p.tiles = a.tiles;
  p.runs = a.runs;
  p.o = a.o;
  p.lse = a.lse;
  p.out_map = a.out_map;
  p.ws = a.ws;
  p.lse_ld = a.lse_ld;
  p.n_tiles = a.n_tiles;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.thresh_raw = 8.0f / p.scale_log2;
  const int64_t items = (int64_t)a.n_tiles * a.H;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffff) {
    *err = "too many query tiles";
    return cudaErrorInvalidValue;
  }
  // persistent blocks, two per SM, each walking items blockIdx.x, +gridDim.x, ...
  const int64_t blocks = std::min<int64_t>(items, 2 * (int64_t)num_sms());
  // Item groups: the smallest divisor of Hkv whose work per block is at least
  // 1.25 times the longest item, so that the last group's longest items do
  // not run alone at the end, as long as the group's K and V fit the budget;
  // past the budget, the largest divisor that fits.
  p.kv_group = 1;
  const int64_t kv_head_bytes = 2 * (int64_t)a.kv_rows_total * a.D * 2;
  const int G = a.H / a.Hkv;
  for (int d = 1; d <= a.Hkv; ++d) {
    if (a.Hkv % d != 0) continue;
    if (d > 1 && d * kv_head_bytes > kKvGroupBytes) break;
    p.kv_group = d;
    if (4 * (int64_t)d * G * a.total_pieces >= 5 * (int64_t)a.max_pieces * blocks) break;
  }
  if (a.D == 128) return a.partial ? launch_tc<128, true>(p, (int)blocks, a.stream)
                                   : launch_tc<128, false>(p, (int)blocks, a.stream);
  return a.partial ? launch_tc<64, true>(p, (int)blocks, a.stream) : launch_tc<64, false>(p, (int)blocks, a.stream);
}

}  // namespace cpattn
