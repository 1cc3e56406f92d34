// Work-list records shared by the host planner and the attention kernels.
//
// A q tile is up to tile_m consecutive query rows of one sequence: inside one
// rank's shard for a ring step, or, for a whole forward call on global rows,
// cut from the sequence's end so that it may hold the end of one chunk and
// the start of the next (owned then by the rank of its last row).  Its KV
// runs list, in ring order, the key rows of the same sequence that the tile's
// queries may see: at ring step t the q rank r reads the shard of rank
// (r - t) mod cp, one run per contiguous piece of it; the position mask inside
// a run leaves each row the pairs of its own ring steps.
#pragma once

#include <stdint.h>

#define CPATTN_WS_HEADER_BYTES 256

#ifdef __cplusplus
namespace cpattn {
#endif

typedef struct QTile {
  int32_t q_row0;     // row of the first query in the Q buffer
  int32_t q_pos0;     // its position inside the sequence
  int32_t out_row0;   // output row of the first query (global, rank-local or gathered)
  int32_t q_rows;     // valid rows, 1..tile_m
  int32_t run_begin;  // KV runs [run_begin, run_end)
  int32_t run_end;
  int32_t n_kv_tiles; // sum over runs of ceil(kv_len / tile_n)
  int32_t rank;       // virtual rank that owns the tile (of its last row)
} QTile;

typedef struct KvRun {
  int32_t kv_row0;    // row of the first key in the K/V buffers
  int32_t kv_pos0;    // its position inside the sequence
  int32_t kv_len;     // keys in the run (>= 1)
  int32_t causal;     // 1: some key may follow some query of the tile (apply the position mask)
} KvRun;

// Fault word at the start of every workspace.
typedef struct WsHeader {
  uint32_t fault;     // 0 = none; else a CPATTN_FAULT_* code
  uint32_t info;      // where (block index)
  uint32_t detail;    // which wait / value
  uint32_t next_item; // work counter of persistent kernels (items handed out beyond the first wave)
  uint32_t wait_limit_us;  // fault-path test support: limit of every bounded wait (0 = the default)
  uint32_t withhold;       // fault-path test support: 1 = the forward's block 0 never loads its first V tile
  uint32_t pad[58];
} WsHeader;

#ifdef __cplusplus
}  // namespace cpattn
#endif

#define CPATTN_FAULT_WAIT_TIMEOUT 1u
