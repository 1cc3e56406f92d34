// Host planner: context-parallel splits, ring schedule and kernel work lists.
#pragma once

#include <cstdint>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/cpattn.h"
#include "worklist.h"

namespace cpattn {

// A run of consecutive global rows of one sequence, owned by one rank.
struct Segment {
  int64_t row0;   // first row (global THD row, or gathered row for GRID2D work lists)
  int64_t len;
  int32_t seq;
  int64_t pos0;   // position of row0 inside its sequence
};

struct WorkList {
  std::vector<QTile> tiles;
  std::vector<KvRun> runs;
  int64_t total_kv_tiles = 0;
};

struct WorkKey {
  int causal, tile_m, tile_n, pair, q_rank, step;  // q_rank = -1: every rank, every step
  int bwd = 0;                                     // 1: backward work list (KV tiles with query runs)
  bool operator<(const WorkKey& o) const {
    return std::tie(bwd, causal, tile_m, tile_n, pair, q_rank, step) <
           std::tie(o.bwd, o.causal, o.tile_m, o.tile_n, o.pair, o.q_rank, o.step);
  }
};

}  // namespace cpattn

struct cpattn_plan {
  int32_t mode = 0;
  int32_t cp = 1;
  int32_t n_seqs = 0;
  int64_t T = 0;
  int32_t split_h = 0, split_w = 0;
  std::vector<int32_t> cu;                 // [n+1]
  std::vector<int64_t> chunk_offsets;      // [n_chunks+1]
  std::vector<int32_t> chunk_ranks;        // [n_chunks]
  std::vector<int64_t> rank_offsets;       // [cp+1]
  std::vector<int32_t> local_cu;           // [cp*(n+1)]
  std::vector<int64_t> index_map;          // [T]
  std::vector<std::vector<cpattn::Segment>> rank_segments;  // per rank, local order
  // ULYSSES2D: the r ring shards after the all-to-all, as segments of the
  // head-sharded buffer (rows in index-map order), and the all-to-all gather map.
  std::vector<std::vector<cpattn::Segment>> ring_segments;
  std::vector<int64_t> a2a_map;            // [u*T]
  // PAIRED: per sample s and time chunk j (index s*tf_chunks + j), the clean
  // and the noisy chunk as segments of the head-sharded buffer.
  int32_t tf_chunks = 0;
  std::vector<cpattn::Segment> tf_clean, tf_noisy;

  std::mutex mu;
  std::map<cpattn::WorkKey, std::shared_ptr<const cpattn::WorkList>> cache;
};

namespace cpattn {

// Returns an empty string on success, else the reason the inputs are invalid.
std::string build_plan(const int32_t* cu, int32_t n_seqs, int32_t cp, int32_t mode,
                       const int32_t* grid_fhw, cpattn_plan_t* out);

void optimal_split(int32_t cp, int32_t* a, int32_t* b);

// Ring schedule entry for (q rank r, step t).  Returns false for causal GRID2D.
bool ring_entry(const cpattn_plan_t& p, int r, int t, bool causal, int32_t* kv_rank, int32_t* kind);

// Work list of q tiles (tile_m rows) with their KV runs in ring order.
// q_rank < 0: all ranks and all steps (whole forward); else one (rank, step).
// Each run is cut into pieces of tile_n keys; with `pair`, two consecutive
// pieces (possibly from different runs) form one KV tile of the kernel.
std::shared_ptr<const WorkList> get_worklist(cpattn_plan_t& p, bool causal, int tile_m, int tile_n, bool pair,
                                             int q_rank, int step);

// Backward work list: the forward's pairs seen from the keys.  Each record of
// `tiles` is a KV tile of up to tile_k consecutive key rows of one sequence
// inside one rank's shard (q_row0/q_pos0/q_rows/out_row0 hold the key rows);
// its runs list, in ring order, the query rows that see it: the KV shard of
// rank k visits q rank (k + t) mod cp at ring step t.  A run starts at the
// first query that sees the tile's first key (causal) and is flagged when some
// of its queries precede some of the tile's keys.  n_kv_tiles holds the number
// of tile_q-query pieces of the runs.  q_rank >= 0 keeps only the pairs of
// ring step `step` of that q rank.
std::shared_ptr<const WorkList> get_worklist_bwd(cpattn_plan_t& p, bool causal, int tile_k, int tile_q, int q_rank,
                                                 int step);

}  // namespace cpattn
