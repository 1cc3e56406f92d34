// Context-parallel planner (host, integer-only).
//
// ZIGZAG: the load-balanced ring split named ZIGZAG-RINGATTN (LongVILA news
//   article, Fig. 5 and Table 2): each sequence is cut into 2*cp chunks and
//   rank r keeps chunks r and 2cp-1-r, so that under a causal mask every rank
//   holds one cheap early chunk and one expensive late chunk.
// GRID2D: LongCat-Video's 2-D split of a latent by height pieces, then width
//   pieces, with the closest-to-square factorisation of cp (tensor split
//   strategy, get_optimal_split).
// CONTIGUOUS: even contiguous token ranges (token stage of LongVILA MM-SP,
//   "Scaling video training with parallelism", section 3, Fig. 2).
// PAIRED: LongLive-2.0's balanced SP ("Scaling video training with
//   parallelism", section 4): each sample is [clean ; noisy] over N time
//   chunks, rank k keeps the clean/noisy pairs of its time chunks, and after
//   the Ulysses all-to-all the teacher-forcing mask (clean chunk j sees clean
//   chunks <= j; noisy chunk j sees clean chunks < j and itself) is applied
//   at chunk granularity by the work list.
// ULYSSES2D: LongVILA's 2D-Attention mesh of u Ulysses (all-to-all) x r ring
//   (P2P) ranks (news article, 2D attention parallelism, Fig. 3 left): zigzag
//   over the ring dimension, each ring shard's rows cut into u contiguous
//   pieces; the all-to-all regroups them by head.
#include "plan.hpp"

#include <algorithm>
#include <cstdio>
#include <iterator>
#include <numeric>

#include "../../include/cpattn.h"

namespace cpattn {

void optimal_split(int32_t cp, int32_t* a, int32_t* b) {
  int32_t s = 1;
  while ((int64_t)(s + 1) * (s + 1) <= cp) ++s;
  while (s > 1 && cp % s != 0) --s;
  *a = s;
  *b = cp / s;
}

// Pieces of ceil(n/parts) with the remainder last (torch split(size) rule).
static bool split_pieces(int64_t n, int32_t parts, std::vector<int64_t>* out) {
  out->clear();
  const int64_t size = (n + parts - 1) / parts;
  for (int64_t left = n; left > 0; left -= size) out->push_back(std::min(size, left));
  return (int64_t)out->size() == parts;
}

static void finish_common(cpattn_plan_t* p) {
  // rank offsets and local cu_seqlens from the per-rank segments
  const int cp = p->cp, n = p->n_seqs;
  p->rank_offsets.assign(cp + 1, 0);
  p->local_cu.assign((size_t)cp * (n + 1), 0);
  p->index_map.clear();
  p->index_map.reserve(p->T);
  for (int r = 0; r < cp; ++r) {
    int64_t count = 0;
    std::vector<int64_t> per_seq(n, 0);
    for (const Segment& s : p->rank_segments[r]) {
      for (int64_t i = 0; i < s.len; ++i) p->index_map.push_back(s.row0 + i);
      per_seq[s.seq] += s.len;
      count += s.len;
    }
    p->rank_offsets[r + 1] = p->rank_offsets[r] + count;
    int32_t* lc = &p->local_cu[(size_t)r * (n + 1)];
    for (int s = 0; s < n; ++s) lc[s + 1] = lc[s] + (int32_t)per_seq[s];
  }
}

// The Ulysses all-to-all as one row gather: head-sharded row i*T + q holds
// source row index_map[q]*u + i of the [T*u, H/u*D] view.
static void build_a2a(cpattn_plan_t* p, int u) {
  p->a2a_map.resize((size_t)u * p->T);
  for (int i = 0; i < u; ++i)
    for (int64_t q = 0; q < p->T; ++q) p->a2a_map[(size_t)i * p->T + q] = p->index_map[q] * u + i;
}

std::string build_plan(const int32_t* cu, int32_t n_seqs, int32_t cp, int32_t mode,
                       const int32_t* grid, cpattn_plan_t* p) {
  if (!cu) return "cu_seqlens is NULL";
  if (n_seqs < 1) return "n_seqs must be >= 1";
  if (cp < 1 || cp > 4096) return "cp_size must be in [1, 4096]";
  if (cu[0] != 0) return "cu_seqlens[0] must be 0";
  for (int s = 0; s < n_seqs; ++s)
    if (cu[s + 1] <= cu[s]) return "cu_seqlens must be strictly increasing";
  p->mode = mode;
  p->cp = cp;
  p->n_seqs = n_seqs;
  p->T = cu[n_seqs];
  p->cu.assign(cu, cu + n_seqs + 1);
  p->rank_segments.assign(cp, {});
  p->chunk_offsets.clear();
  p->chunk_ranks.clear();
  p->split_h = p->split_w = 0;

  if (mode == CPATTN_MODE_ZIGZAG) {
    const int C = 2 * cp;
    for (int s = 0; s < n_seqs; ++s) {
      const int64_t L = (int64_t)cu[s + 1] - cu[s];
      if (L < C) return "zigzag needs every sequence to have at least 2*cp tokens";
      const int64_t base = L / C, rem = L % C;
      std::vector<int64_t> start(C + 1);
      start[0] = cu[s];
      for (int j = 0; j < C; ++j) start[j + 1] = start[j] + base + (j < rem ? 1 : 0);
      for (int j = 0; j < C; ++j) {
        p->chunk_offsets.push_back(start[j]);
        p->chunk_ranks.push_back(j < cp ? j : C - 1 - j);
      }
      for (int r = 0; r < cp; ++r) {
        const int lo = r, hi = C - 1 - r;
        p->rank_segments[r].push_back({start[lo], start[lo + 1] - start[lo], s, start[lo] - cu[s]});
        p->rank_segments[r].push_back({start[hi], start[hi + 1] - start[hi], s, start[hi] - cu[s]});
      }
    }
    p->chunk_offsets.push_back(p->T);
  } else if (mode == CPATTN_MODE_GRID2D) {
    if (!grid) return "grid2d needs a grid";
    if (n_seqs != 1) return "grid2d plans one latent (n_seqs must be 1)";
    const int64_t F = grid[0], h = grid[1], w = grid[2];
    if (F < 1 || h < 1 || w < 1 || F * h * w != p->T) return "grid frames*height*width must equal T";
    int32_t a, b;
    optimal_split(cp, &a, &b);
    const int32_t sh = (h > w) ? b : a, sw = (h > w) ? a : b;
    std::vector<int64_t> hp, wp;
    if (!split_pieces(h, sh, &hp)) return "height cannot be cut into split_h pieces";
    if (!split_pieces(w, sw, &wp)) return "width cannot be cut into split_w pieces";
    p->split_h = sh;
    p->split_w = sw;
    std::vector<int64_t> h0(sh + 1, 0), w0(sw + 1, 0);
    for (int i = 0; i < sh; ++i) h0[i + 1] = h0[i] + hp[i];
    for (int i = 0; i < sw; ++i) w0[i + 1] = w0[i] + wp[i];
    // rank tiles, (f, y, x) row-major inside each tile
    for (int ih = 0; ih < sh; ++ih)
      for (int iw = 0; iw < sw; ++iw) {
        auto& segs = p->rank_segments[ih * sw + iw];
        for (int64_t f = 0; f < F; ++f)
          for (int64_t y = h0[ih]; y < h0[ih + 1]; ++y) {
            const int64_t row = f * h * w + y * w + w0[iw];
            segs.push_back({row, wp[iw], 0, row});
          }
      }
    // chunks: (frame, row, w-piece) runs in global order
    for (int64_t f = 0; f < F; ++f)
      for (int64_t y = 0; y < h; ++y) {
        const int ih = (int)(std::upper_bound(h0.begin(), h0.end(), y) - h0.begin()) - 1;
        for (int iw = 0; iw < sw; ++iw) {
          p->chunk_offsets.push_back(f * h * w + y * w + w0[iw]);
          p->chunk_ranks.push_back(ih * sw + iw);
        }
      }
    p->chunk_offsets.push_back(p->T);
  } else if (mode == CPATTN_MODE_CONTIGUOUS) {
    if (p->T < cp) return "contiguous split needs at least cp tokens";
    const int64_t q = p->T / cp, rem = p->T % cp;
    int64_t start = 0;
    int s = 0;
    for (int r = 0; r < cp; ++r) {
      const int64_t len = q + (r < rem ? 1 : 0), end = start + len;
      p->chunk_offsets.push_back(start);
      p->chunk_ranks.push_back(r);
      for (int64_t a = start; a < end;) {
        while (cu[s + 1] <= a) ++s;
        const int64_t b = std::min<int64_t>(end, cu[s + 1]);
        p->rank_segments[r].push_back({a, b - a, s, a - cu[s]});
        a = b;
      }
      start = end;
    }
    p->chunk_offsets.push_back(p->T);
  } else if (mode == CPATTN_MODE_ULYSSES2D) {
    if (!grid) return "ulysses2d needs the mesh";
    const int32_t u = grid[0], r = grid[1];
    if (u < 1 || r < 1 || (int64_t)u * r != cp) return "cp must equal ulysses * ring";
    const int C = 2 * r;
    // ring shards: zigzag over r, local order chunk j then chunk C-1-j of each sequence
    std::vector<std::vector<Segment>> ring(r);
    for (int s = 0; s < n_seqs; ++s) {
      const int64_t L = (int64_t)cu[s + 1] - cu[s];
      if (L < C) return "ulysses2d needs every sequence to have at least 2*ring tokens";
      const int64_t base = L / C, rem = L % C;
      std::vector<int64_t> start(C + 1);
      start[0] = cu[s];
      for (int j = 0; j < C; ++j) start[j + 1] = start[j] + base + (j < rem ? 1 : 0);
      for (int j = 0; j < r; ++j) {
        ring[j].push_back({start[j], start[j + 1] - start[j], s, start[j] - cu[s]});
        ring[j].push_back({start[C - 1 - j], start[C - j] - start[C - 1 - j], s, start[C - 1 - j] - cu[s]});
      }
    }
    // the u Ulysses ranks of ring group j hold u contiguous pieces of its local rows
    for (int j = 0; j < r; ++j) {
      int64_t Tj = 0;
      for (const Segment& sg : ring[j]) Tj += sg.len;
      if (Tj < u) return "a ring shard has fewer tokens than the Ulysses degree";
      const int64_t q = Tj / u, rem = Tj % u;
      size_t si = 0;
      int64_t used = 0;  // rows of ring[j][si] already handed out
      for (int i = 0; i < u; ++i) {
        int64_t need = q + (i < rem ? 1 : 0);
        auto& dst = p->rank_segments[(size_t)j * u + i];
        while (need > 0) {
          const Segment& sg = ring[j][si];
          const int64_t take = std::min(need, sg.len - used);
          dst.push_back({sg.row0 + used, take, sg.seq, sg.pos0 + used});
          used += take;
          need -= take;
          if (used == sg.len) {
            ++si;
            used = 0;
          }
        }
      }
    }
    p->split_h = u;
    p->split_w = r;
    finish_common(p);
    // chunks: maximal runs of consecutive global rows of one sequence owned by one rank
    std::vector<int32_t> owner(p->T);
    for (int g = 0; g < cp; ++g)
      for (const Segment& sg : p->rank_segments[g])
        for (int64_t t = 0; t < sg.len; ++t) owner[sg.row0 + t] = g;
    int s = 0;
    for (int64_t t = 0; t < p->T; ++t) {
      bool new_seq = false;
      while (cu[s + 1] <= t) {
        ++s;
        new_seq = true;
      }
      if (t == 0 || owner[t] != owner[t - 1] || new_seq) {
        p->chunk_offsets.push_back(t);
        p->chunk_ranks.push_back(owner[t]);
      }
    }
    p->chunk_offsets.push_back(p->T);
    // after the all-to-all: ring shard j is rows [rank_offsets[j*u], rank_offsets[(j+1)*u]) of
    // each head group's buffer, in its zigzag local order
    p->ring_segments.assign(r, {});
    for (int j = 0; j < r; ++j) {
      int64_t row = p->rank_offsets[(size_t)j * u];
      for (const Segment& sg : ring[j]) {
        p->ring_segments[j].push_back({row, sg.len, sg.seq, sg.pos0});
        row += sg.len;
      }
    }
    build_a2a(p, u);
    return std::string();
  } else if (mode == CPATTN_MODE_PAIRED) {
    if (!grid) return "paired plans need the number of time chunks";
    const int32_t N = grid[0];
    if (N < 1 || N % cp != 0) return "the number of time chunks must be a positive multiple of cp";
    const int32_t m = N / cp;
    // per sample: [clean ; noisy], each stream in N chunks of floor(half/N) + [j < half mod N] tokens
    std::vector<int64_t> cstart((size_t)n_seqs * (N + 1)), nstart((size_t)n_seqs * (N + 1));
    for (int s = 0; s < n_seqs; ++s) {
      const int64_t L = (int64_t)cu[s + 1] - cu[s];
      if (L % 2 != 0 || L / 2 < N) return "paired samples need an even length with at least N tokens per stream";
      const int64_t half = L / 2;
      int64_t* cs = &cstart[(size_t)s * (N + 1)];
      int64_t* ns = &nstart[(size_t)s * (N + 1)];
      cs[0] = cu[s];
      ns[0] = cu[s] + half;
      for (int j = 0; j < N; ++j) {
        const int64_t sz = half / N + (j < half % N ? 1 : 0);
        cs[j + 1] = cs[j] + sz;
        ns[j + 1] = ns[j] + sz;
      }
      for (int j = 0; j < N; ++j) {
        auto& dst = p->rank_segments[(size_t)(j / m)];
        dst.push_back({cs[j], cs[j + 1] - cs[j], s, cs[j] - cu[s]});
        dst.push_back({ns[j], ns[j + 1] - ns[j], s, ns[j] - cu[s]});
      }
      // chunks in global order: the clean chunks, then the noisy chunks
      for (int j = 0; j < N; ++j) {
        p->chunk_offsets.push_back(cs[j]);
        p->chunk_ranks.push_back(j / m);
      }
      for (int j = 0; j < N; ++j) {
        p->chunk_offsets.push_back(ns[j]);
        p->chunk_ranks.push_back(j / m);
      }
    }
    p->chunk_offsets.push_back(p->T);
    p->split_h = cp;  // a Ulysses layout over all cp ranks with one ring group
    p->split_w = 1;
    finish_common(p);
    // the clean and noisy chunks in the head-sharded buffer (rows in index-map order)
    p->tf_chunks = N;
    p->tf_clean.assign((size_t)n_seqs * N, {});
    p->tf_noisy.assign((size_t)n_seqs * N, {});
    std::vector<int64_t> row(cp);
    for (int k = 0; k < cp; ++k) row[k] = p->rank_offsets[k];
    for (int s = 0; s < n_seqs; ++s)
      for (int j = 0; j < N; ++j) {
        const int64_t* cs = &cstart[(size_t)s * (N + 1)];
        const int64_t* ns = &nstart[(size_t)s * (N + 1)];
        int64_t& r = row[j / m];
        p->tf_clean[(size_t)s * N + j] = {r, cs[j + 1] - cs[j], s, cs[j] - cu[s]};
        r += cs[j + 1] - cs[j];
        p->tf_noisy[(size_t)s * N + j] = {r, ns[j + 1] - ns[j], s, ns[j] - cu[s]};
        r += ns[j + 1] - ns[j];
      }
    build_a2a(p, cp);
    return std::string();
  } else {
    return "unknown mode";
  }
  finish_common(p);
  return std::string();
}

bool ring_entry(const cpattn_plan_t& p, int r, int t, bool causal, int32_t* kv_rank, int32_t* kind) {
  if (p.mode == CPATTN_MODE_ULYSSES2D || p.mode == CPATTN_MODE_PAIRED) {
    // after the all-to-all, rank (i, j) rings over the r ring groups with its head group
    // (PAIRED: one ring group, every key local after the all-to-all)
    const int u = p.split_h, nr = p.split_w, i = r % u, j = r / u;
    if (t >= nr) {
      *kv_rank = -1;
      *kind = CPATTN_MASK_SKIP;
      return true;
    }
    const int k = ((j - t) % nr + nr) % nr;
    *kv_rank = k * u + i;
    *kind = !causal ? CPATTN_MASK_FULL : (k == j ? CPATTN_MASK_DIAG : (k < j ? CPATTN_MASK_KV_HEAD : CPATTN_MASK_Q_TAIL));
    return true;
  }
  const int cp = p.cp;
  const int k = ((r - t) % cp + cp) % cp;
  *kv_rank = k;
  if (!causal) {
    *kind = CPATTN_MASK_FULL;
  } else if (k == r) {
    *kind = CPATTN_MASK_DIAG;
  } else if (p.mode == CPATTN_MODE_ZIGZAG) {
    *kind = (k < r) ? CPATTN_MASK_KV_HEAD : CPATTN_MASK_Q_TAIL;
  } else if (p.mode == CPATTN_MODE_CONTIGUOUS) {
    *kind = (k < r) ? CPATTN_MASK_FULL : CPATTN_MASK_SKIP;
  } else {
    return false;
  }
  return true;
}

// Appends a run to a tile's list; a run that continues the previous run of
// the same ring step (the next rows and positions of the same shard) is
// merged into it, masked if either part is.
static void append_run(WorkList* wl, size_t step_begin, const KvRun& run) {
  if (wl->runs.size() > step_begin) {
    KvRun& prev = wl->runs.back();
    if (prev.kv_row0 + prev.kv_len == run.kv_row0 && prev.kv_pos0 + prev.kv_len == run.kv_pos0) {
      prev.kv_len += run.kv_len;
      prev.causal |= run.causal;
      return;
    }
  }
  wl->runs.push_back(run);
}

// Segments of `rank` that belong to sequence `seq` (segments are ordered by sequence).
static std::pair<size_t, size_t> seq_range(const std::vector<Segment>& segs, int32_t seq) {
  auto lo = std::lower_bound(segs.begin(), segs.end(), seq,
                             [](const Segment& s, int32_t v) { return s.seq < v; });
  auto hi = std::upper_bound(segs.begin(), segs.end(), seq,
                             [](int32_t v, const Segment& s) { return v < s.seq; });
  return {(size_t)(lo - segs.begin()), (size_t)(hi - segs.begin())};
}

// Replicates a work list over the u head groups of a head-sharded buffer
// (group i's rows start at i*T).
static void replicate_head_groups(const cpattn_plan_t& p, WorkList* wl) {
  const size_t nt = wl->tiles.size(), nr = wl->runs.size();
  const int u = p.split_h;
  for (int i = 1; i < u; ++i) {
    const int32_t off = (int32_t)(i * p.T);
    for (size_t t = 0; t < nt; ++t) {
      QTile c = wl->tiles[t];
      c.q_row0 += off;
      c.out_row0 += off;
      c.run_begin += (int32_t)(i * nr);
      c.run_end += (int32_t)(i * nr);
      wl->tiles.push_back(c);
    }
    for (size_t q = 0; q < nr; ++q) {
      KvRun c = wl->runs[q];
      c.kv_row0 += off;
      wl->runs.push_back(c);
    }
  }
  wl->total_kv_tiles *= u;
}

// PAIRED: the teacher-forcing mask at chunk granularity; every run is fully visible.
static std::shared_ptr<WorkList> build_worklist_paired(const cpattn_plan_t& p, int tile_m, int tile_n, bool pair) {
  auto wl = std::make_shared<WorkList>();
  const int N = p.tf_chunks;
  for (int s = 0; s < p.n_seqs; ++s)
    for (int j = 0; j < N; ++j)
      for (int noisy = 0; noisy < 2; ++noisy) {
        const Segment& qs = noisy ? p.tf_noisy[(size_t)s * N + j] : p.tf_clean[(size_t)s * N + j];
        std::vector<Segment> keys;
        for (int jj = 0; jj < (noisy ? j : j + 1); ++jj) keys.push_back(p.tf_clean[(size_t)s * N + jj]);
        if (noisy) keys.push_back(qs);
        for (int64_t off = 0; off < qs.len; off += tile_m) {
          QTile t{};
          const int64_t rows = std::min<int64_t>(tile_m, qs.len - off);
          t.q_row0 = (int32_t)(qs.row0 + off);
          t.q_pos0 = (int32_t)(qs.pos0 + off);
          t.q_rows = (int32_t)rows;
          t.out_row0 = t.q_row0;
          t.rank = j / (N / p.cp);
          t.run_begin = (int32_t)wl->runs.size();
          int64_t ntiles = 0;
          for (const Segment& ks : keys) {
            wl->runs.push_back({(int32_t)ks.row0, (int32_t)ks.pos0, (int32_t)ks.len, 0});
            ntiles += (ks.len + tile_n - 1) / tile_n;
          }
          t.run_end = (int32_t)wl->runs.size();
          if (pair) ntiles = (ntiles + 1) / 2;
          t.n_kv_tiles = (int32_t)ntiles;
          wl->total_kv_tiles += ntiles;
          wl->tiles.push_back(t);
        }
      }
  replicate_head_groups(p, wl.get());
  std::stable_sort(wl->tiles.begin(), wl->tiles.end(),
                   [](const QTile& a, const QTile& b) { return a.n_kv_tiles > b.n_kv_tiles; });
  return wl;
}

static std::shared_ptr<WorkList> build_worklist(const cpattn_plan_t& p, bool causal, int tile_m,
                                                int tile_n, bool pair, int q_rank, int step) {
  if (p.mode == CPATTN_MODE_PAIRED) return build_worklist_paired(p, tile_m, tile_n, pair);
  auto wl = std::make_shared<WorkList>();
  const bool mesh = (p.mode == CPATTN_MODE_ULYSSES2D);  // (PAIRED returned above)
  const int cp = mesh ? p.split_w : p.cp;
  const bool gathered = (p.mode == CPATTN_MODE_GRID2D);
  // For GRID2D the kernel reads gathered shards: rank r's rows are the
  // contiguous range [rank_offsets[r], rank_offsets[r+1]) of the gathered buffers.
  // For ULYSSES2D it reads the head-sharded buffers of the all-to-all, whose
  // ring shards are p.ring_segments.
  auto segments_of = [&](int r) {
    if (mesh) return p.ring_segments[r];
    if (!gathered) return p.rank_segments[r];
    std::vector<Segment> one;
    const int64_t a = p.rank_offsets[r], b = p.rank_offsets[r + 1];
    if (b > a) one.push_back({a, b - a, 0, a});
    return one;
  };
  std::vector<std::vector<Segment>> segs(cp);
  for (int r = 0; r < cp; ++r) segs[r] = segments_of(r);

  // The KV runs a query tile [qp_first, qp_last] of sequence `seq` owned by
  // rank r reads at ring steps [s_lo, s_hi): at step st the pieces of rank
  // (r - st) mod cp's shard of the sequence; runs in the future are dropped,
  // runs crossing the diagonal are cut at the tile's last query and masked.
  auto add_runs = [&](QTile* t, int r, int32_t seq, int64_t qp_first, int64_t qp_last, int s_lo, int s_hi) {
    t->run_begin = (int32_t)wl->runs.size();
    for (int st = s_lo; st < s_hi; ++st) {
      const int k = ((r - st) % cp + cp) % cp;
      const auto rng = seq_range(segs[k], seq);
      const size_t step_begin = wl->runs.size();
      for (size_t i = rng.first; i < rng.second; ++i) {
        const Segment& ks = segs[k][i];
        KvRun run{};
        run.kv_row0 = (int32_t)ks.row0;
        run.kv_pos0 = (int32_t)ks.pos0;
        int64_t len = ks.len;
        run.causal = 0;
        if (causal) {
          if (ks.pos0 > qp_last) continue;                   // entirely in the future
          if (ks.pos0 + ks.len - 1 > qp_first) {             // crosses the diagonal
            len = std::min<int64_t>(ks.len, qp_last - ks.pos0 + 1);
            run.causal = 1;
          }
        }
        run.kv_len = (int32_t)len;
        append_run(wl.get(), step_begin, run);
      }
    }
    t->run_end = (int32_t)wl->runs.size();
    int64_t ntiles = 0;
    for (int32_t i = t->run_begin; i < t->run_end; ++i) ntiles += (wl->runs[i].kv_len + tile_n - 1) / tile_n;
    if (pair) ntiles = (ntiles + 1) / 2;  // two pieces per kernel tile
    t->n_kv_tiles = (int32_t)ntiles;
    wl->total_kv_tiles += ntiles;
  };

  if (q_rank < 0 && !mesh && !gathered) {
    // Whole call on global rows (zigzag, contiguous): a sequence's query rows
    // are consecutive, so its tiles are cut from the sequence itself, ending
    // at its last row (a partial tile falls at the start, where it sees the
    // fewest keys), and a tile may hold the end of one chunk and the start of
    // the next.  Each row still sees its own keys shard by shard: the tile
    // walks the ring of the rank that owns its last row, and the position
    // mask inside every run that crosses the tile's first query leaves each
    // row exactly the pairs of its own ring steps.
    std::vector<std::vector<std::pair<int64_t, int>>> owner(p.n_seqs);  // (pos0, rank) of each segment
    std::vector<int64_t> base(p.n_seqs, -1), len(p.n_seqs, 0);
    for (int r = 0; r < cp; ++r)
      for (const Segment& qs : segs[r]) {
        owner[qs.seq].push_back({qs.pos0, r});
        base[qs.seq] = qs.row0 - qs.pos0;
        len[qs.seq] += qs.len;
      }
    for (int32_t sq = 0; sq < p.n_seqs; ++sq) {
      std::sort(owner[sq].begin(), owner[sq].end());
      for (int64_t end = len[sq]; end > 0; end -= tile_m) {
        const int64_t first = std::max<int64_t>(0, end - tile_m);
        // the segment holding the last row: the last one starting at or before it
        auto it = std::upper_bound(owner[sq].begin(), owner[sq].end(), std::make_pair(end - 1, cp));
        const int r = std::prev(it)->second;
        QTile t{};
        t.q_row0 = (int32_t)(base[sq] + first);
        t.q_pos0 = (int32_t)first;
        t.q_rows = (int32_t)(end - first);
        t.rank = r;
        t.out_row0 = t.q_row0;
        add_runs(&t, r, sq, first, end - 1, 0, cp);
        wl->tiles.push_back(t);
      }
    }
  }
  const int r_lo = q_rank < 0 ? 0 : q_rank, r_hi = (q_rank < 0 ? (mesh || gathered ? cp : 0) : q_rank + 1);
  for (int r = r_lo; r < r_hi; ++r) {
    int64_t local = 0;  // rank-local row of the current segment
    for (const Segment& qs : segs[r]) {
      for (int64_t off = 0; off < qs.len; off += tile_m) {
        QTile t{};
        const int64_t rows = std::min<int64_t>(tile_m, qs.len - off);
        t.q_row0 = (int32_t)(qs.row0 + off);
        t.q_pos0 = (int32_t)(qs.pos0 + off);
        t.q_rows = (int32_t)rows;
        t.rank = r;
        if (q_rank >= 0)
          t.out_row0 = (int32_t)(local + off);  // partial outputs: rank-local rows
        else
          t.out_row0 = t.q_row0;                // global rows (gathered rows for GRID2D)
        const int64_t qp_first = qs.pos0 + off, qp_last = qp_first + rows - 1;
        add_runs(&t, r, qs.seq, qp_first, qp_last, q_rank < 0 ? 0 : step, q_rank < 0 ? cp : step + 1);
        wl->tiles.push_back(t);
      }
      local += qs.len;
    }
  }
  if (mesh) replicate_head_groups(p, wl.get());  // one copy of the ring work per head group
  // Longest tiles first, so that the block scheduler's in-order dispatch
  // finishes the heaviest work early (LPT order).
  std::stable_sort(wl->tiles.begin(), wl->tiles.end(),
                   [](const QTile& a, const QTile& b) { return a.n_kv_tiles > b.n_kv_tiles; });
  return wl;
}

std::shared_ptr<const WorkList> get_worklist(cpattn_plan_t& p, bool causal, int tile_m, int tile_n, bool pair,
                                             int q_rank, int step) {
  WorkKey key{causal ? 1 : 0, tile_m, tile_n, pair ? 1 : 0, q_rank, step};
  std::lock_guard<std::mutex> lock(p.mu);
  auto it = p.cache.find(key);
  if (it != p.cache.end()) return it->second;
  auto wl = build_worklist(p, causal, tile_m, tile_n, pair, q_rank, step);
  p.cache[key] = wl;
  return wl;
}

}  // namespace cpattn

namespace cpattn {

static std::shared_ptr<WorkList> build_worklist_bwd(const cpattn_plan_t& p, bool causal, int tile_k, int tile_q,
                                                    int q_rank, int step) {
  auto wl = std::make_shared<WorkList>();
  const int cp = p.cp;
  const bool gathered = (p.mode == CPATTN_MODE_GRID2D);
  std::vector<std::vector<Segment>> segs(cp);
  for (int r = 0; r < cp; ++r) {
    if (!gathered) {
      segs[r] = p.rank_segments[r];
    } else {
      const int64_t a = p.rank_offsets[r], b = p.rank_offsets[r + 1];
      if (b > a) segs[r].push_back({a, b - a, 0, a});
    }
  }
  // The query runs a KV tile [kp_first, kp_last] of sequence `seq` meets at
  // the q ranks `q_ranks` (in ring order): queries before the tile's first
  // key see none of it; runs with a query before the tile's last key are
  // masked.
  auto add_runs = [&](QTile* t, const std::vector<int>& q_ranks, int32_t seq, int64_t kp_first, int64_t kp_last) {
    t->run_begin = (int32_t)wl->runs.size();
    for (int r : q_ranks) {
      const auto rng = seq_range(segs[r], seq);
      const size_t step_begin = wl->runs.size();
      for (size_t i = rng.first; i < rng.second; ++i) {
        const Segment& qs = segs[r][i];
        int64_t q0 = qs.pos0, q1 = qs.pos0 + qs.len;  // query positions [q0, q1)
        KvRun run{};
        run.causal = 0;
        if (causal) {
          if (q1 - 1 < kp_first) continue;         // every query precedes the tile
          q0 = std::max<int64_t>(q0, kp_first);    // queries before the first key see nothing
          if (q0 < kp_last) run.causal = 1;        // some query precedes some key
        }
        run.kv_row0 = (int32_t)(qs.row0 + (q0 - qs.pos0));
        run.kv_pos0 = (int32_t)q0;
        run.kv_len = (int32_t)(q1 - q0);
        append_run(wl.get(), step_begin, run);
      }
    }
    t->run_end = (int32_t)wl->runs.size();
    int64_t pieces = 0;
    for (int32_t i = t->run_begin; i < t->run_end; ++i) pieces += (wl->runs[i].kv_len + tile_q - 1) / tile_q;
    t->n_kv_tiles = (int32_t)pieces;
    wl->total_kv_tiles += pieces;
  };

  if (q_rank < 0 && !gathered) {
    // Whole call on global rows (zigzag, contiguous): KV tiles are cut from
    // each sequence from its first row on (a partial tile falls at the end,
    // where the fewest queries see it), so a tile may hold the end of one
    // chunk and the start of the next.  It is owned by the rank of its first
    // key and meets the q ranks of that rank's ring; the position mask leaves
    // each key the queries of its own ring steps.
    std::vector<std::vector<std::pair<int64_t, int>>> owner(p.n_seqs);  // (pos0, rank) of each segment
    std::vector<int64_t> base(p.n_seqs, -1), len(p.n_seqs, 0);
    for (int r = 0; r < cp; ++r)
      for (const Segment& ks : segs[r]) {
        owner[ks.seq].push_back({ks.pos0, r});
        base[ks.seq] = ks.row0 - ks.pos0;
        len[ks.seq] += ks.len;
      }
    std::vector<int> q_ranks(cp);
    for (int32_t sq = 0; sq < p.n_seqs; ++sq) {
      std::sort(owner[sq].begin(), owner[sq].end());
      for (int64_t first = 0; first < len[sq]; first += tile_k) {
        const int64_t last = std::min<int64_t>(len[sq], first + tile_k) - 1;
        auto it = std::upper_bound(owner[sq].begin(), owner[sq].end(), std::make_pair(first, cp));
        const int k = std::prev(it)->second;
        QTile t{};
        t.q_row0 = (int32_t)(base[sq] + first);
        t.q_pos0 = (int32_t)first;
        t.q_rows = (int32_t)(last - first + 1);
        t.out_row0 = t.q_row0;
        t.rank = k;
        for (int tt = 0; tt < cp; ++tt) q_ranks[tt] = (k + tt) % cp;
        add_runs(&t, q_ranks, sq, first, last);
        wl->tiles.push_back(t);
      }
    }
  }
  // KV ranks to visit, each with the ring steps (q ranks) that read it
  for (int k = 0; k < (q_rank < 0 && !gathered ? 0 : cp); ++k) {
    std::vector<int> q_ranks;
    if (q_rank < 0) {
      for (int t = 0; t < cp; ++t) q_ranks.push_back((k + t) % cp);
    } else {
      if (((q_rank - step) % cp + cp) % cp != k) continue;
      q_ranks.push_back(q_rank);
    }
    for (const Segment& ks : segs[k]) {
      for (int64_t off = 0; off < ks.len; off += tile_k) {
        QTile t{};
        const int64_t rows = std::min<int64_t>(tile_k, ks.len - off);
        t.q_row0 = (int32_t)(ks.row0 + off);
        t.q_pos0 = (int32_t)(ks.pos0 + off);
        t.q_rows = (int32_t)rows;
        t.out_row0 = t.q_row0;
        t.rank = k;
        const int64_t kp_first = ks.pos0 + off, kp_last = kp_first + rows - 1;
        add_runs(&t, q_ranks, ks.seq, kp_first, kp_last);
        wl->tiles.push_back(t);
      }
    }
  }
  std::stable_sort(wl->tiles.begin(), wl->tiles.end(),
                   [](const QTile& a, const QTile& b) { return a.n_kv_tiles > b.n_kv_tiles; });
  return wl;
}

std::shared_ptr<const WorkList> get_worklist_bwd(cpattn_plan_t& p, bool causal, int tile_k, int tile_q, int q_rank,
                                                 int step) {
  WorkKey key{causal ? 1 : 0, tile_k, tile_q, 0, q_rank, step};
  key.bwd = 1;
  std::lock_guard<std::mutex> lock(p.mu);
  auto it = p.cache.find(key);
  if (it != p.cache.end()) return it->second;
  auto wl = build_worklist_bwd(p, causal, tile_k, tile_q, q_rank, step);
  p.cache[key] = wl;
  return wl;
}

}  // namespace cpattn
