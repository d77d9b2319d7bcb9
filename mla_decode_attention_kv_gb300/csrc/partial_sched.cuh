// Work partition of the partial-attention kernels (16-bit and FP8 caches):
// the units (sequence, query token, part), their 128-token tiles, the share
// of the flat tile sequence each CTA pair takes, the bounded pipeline waits
// and the TMA box rows of a paged tile.
#pragma once
#include <climits>
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

// Token range of one unit.  History shard p of sequence b covers
// [p*len, min(L, (p+1)*len)), len = bs * ceil(L / (S*bs)) (block-aligned,
// trailing shards possibly empty).  The CURRENT part covers kv_cur[b, 0..i].
// Units are numbered u = ((i * B + b) * P + p): the parts of one query token
// are consecutive, so a cluster walking a contiguous range reuses Q; and with
// several query tokens (MTP) the units of token i form the i-th block of the
// order, so the equal shares give the pairs of each block the same KV ranges at
// the same time: the second token's stream finds the KV in L2 (measured with
// two tokens: 306 MB of DRAM reads for 302 MB of cache, against 606 MB with
// the tokens of one sequence next to each other).
struct UnitInfo {
  int b, i, p;
  int lo, hi;
  bool current;
  int ntiles;
};

// (out of line: it is called from every role's tile iterator, rarely on the
// per-tile path, and its inlined copies would spread the kernels' hot loops
// over more instruction-cache lines)
template <int TILE>
__device__ __noinline__ UnitInfo unit_info(const PartialParams& pp, int u) {
  UnitInfo ui;
  ui.p = u % pp.P;
  const int ib = u / pp.P;   // units by query token, then sequence, then part
  ui.b = ib % pp.B;
  ui.i = ib / pp.B;
  ui.current = pp.has_cur && ui.p == pp.S;
  if (ui.current) {
    ui.lo = 0;
    ui.hi = ui.i + 1;
  } else {
    int L = pp.seq_lens[ui.b];
    const int cap = pp.max_blocks * pp.bs;
    if (L < 0 || L > cap) {
      // a history longer than its block-table row (or negative): flagged,
      // then clamped so that no access leaves the table
      set_error(pp.err, kDevBadSeqLen);
      L = max(0, min(L, cap));
    }
    const int chunk = pp.S * pp.bs;
    const int len = L > 0 ? pp.bs * ((L + chunk - 1) / chunk) : 0;
    ui.lo = min(L, ui.p * len);
    ui.hi = min(L, (ui.p + 1) * len);
  }
  ui.ntiles = (ui.hi - ui.lo + TILE - 1) / TILE;
  return ui;
}

// The first units of a pair's range, looked up once when the kernel starts
// (partition_tiles fills the table): every role's tile iterator then reads a
// unit's geometry from shared memory instead of recomputing it, with a
// seq_lens load and integer divisions, on its issue path at each unit
// boundary.  Units past the table are computed as before.
constexpr int kUnitCache = 64;
__shared__ UnitInfo s_unit_cache[kUnitCache];
__shared__ int s_unit_range[2];   // first unit of the table, entries

// (out of line, like unit_info: the iterators' copies stay off the hot loops)
template <int TILE>
__device__ __noinline__ UnitInfo unit_get(const PartialParams& pp, int u) {
  const unsigned k = static_cast<unsigned>(u - s_unit_range[0]);
  if (k < static_cast<unsigned>(s_unit_range[1])) return s_unit_cache[k];
  return unit_info<TILE>(pp, u);
}

// Row of o_part / lse_part holding token t (= b * q_len + i), part p, head h.
// The partials are laid out as head_slices blocks of H / head_slices heads,
// [head_slices][T][P][H / head_slices]; with one slice that is [T][P][H].
// (Slices make each destination's share of a head-scattered all-to-all one
// contiguous block.)
__device__ __forceinline__ int64_t part_row(const PartialParams& pp, int64_t t, int p, int h) {
  const int hs = pp.H / pp.head_slices;
  const int s = h / hs;
  return ((static_cast<int64_t>(s) * pp.T + t) * pp.P + p) * hs + (h - s * hs);
}

// Tile range of one cluster: tiles [j_begin, ...) of unit u_begin through
// tiles [..., j_stop) of unit u_last, in the flat order of the units' tiles
// (global tile index t_begin of the first one).
struct TileRange {
  int u_begin, j_begin, u_last, j_stop, t_begin;
};

// Walks the tiles of a TileRange as one flat stream.  A "piece" is the part
// of one unit inside the range: the whole unit, or (at the ends of the range
// of a cluster that splits units) a run of its tiles.
template <int TILE>
struct TileIter {
  int u, j, k, nq, qkey;
  int jfirst, jend;      // tile bounds of the current piece within its unit
  int ustart;            // global tile index of the unit's first tile
  int u_last, j_stop;
  bool newq, valid;
  UnitInfo ui;
  __device__ __forceinline__ void start(const PartialParams& pp, const TileRange& r) {
    u_last = r.u_last;
    j_stop = r.j_stop;
    k = -1;
    nq = -1;
    qkey = -1;
    valid = r.u_begin <= r.u_last;
    if (!valid) return;
    u = r.u_begin;
    ui = unit_get<TILE>(pp, u);
    ustart = r.t_begin - r.j_begin;
    enter(pp, r.j_begin);
  }
  __device__ __forceinline__ void enter(const PartialParams& pp, int j0) {
    ++k;
    j = jfirst = j0;
    jend = u == u_last ? j_stop : ui.ntiles;
    const int key = ui.b * pp.q_len + ui.i;
    newq = key != qkey;
    if (newq) {
      ++nq;
      qkey = key;
    }
  }
  __device__ __forceinline__ void next_unit(const PartialParams& pp) {
    while (u < u_last) {
      ustart += ui.ntiles;
      ++u;
      ui = unit_get<TILE>(pp, u);
      if (ui.ntiles > 0) {
        enter(pp, 0);
        return;
      }
    }
    valid = false;
  }
  __device__ __forceinline__ void advance(const PartialParams& pp) {
    if (++j >= jend) next_unit(pp);
  }
  __device__ __forceinline__ bool first() const { return j == jfirst; }
  __device__ __forceinline__ bool last() const { return j == jend - 1; }
  // Whether the current piece is the whole unit (no other cluster holds tiles of it).
  __device__ __forceinline__ bool whole() const { return jfirst == 0 && jend == ui.ntiles; }
  // Whether this tile is the last one that reads the current Q.
  __device__ __forceinline__ bool last_of_q(const PartialParams& pp) const {
    if (!last()) return false;
    TileIter n = *this;
    n.next_unit(pp);
    return !n.valid || n.newq;
  }
};

// Tile shares of the CTA pairs: pair c takes tiles [start(c), start(c + 1))
// of the flat order of all units' tiles.  The boundaries are a table made by
// partition_tiles (equal shares of cost, below), kept in shared memory by the
// partial kernels and in the workspace for the merge kernel.
struct Shares {
  const int* bound;   // [ncl + 1], non-decreasing, bound[0] = 0, bound[ncl] = total
  int64_t total;      // tiles of all units
  int ncl;
  __device__ __forceinline__ int64_t start(int c) const { return bound[c]; }
  __device__ __forceinline__ int cluster_of(int64_t t) const {   // the pair whose share holds tile t
    int lo = 0, hi = ncl - 1;   // the last c with start(c) <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bound[mid] <= t)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  }
};

// Cost of a unit for the shares, in half tiles: its tiles, plus half a tile
// for what every piece costs a pair besides its tiles (the restart of the
// pipelines at a new unit, the epilogue).  Measured on GB300 with a batch of
// ragged histories (64 sequences of 512 to 65536 tokens in 16 shards): with
// equal tile shares a pair's finishing time grew by ~1.7 us, about half a
// tile, per piece it held, and the pairs held 3 to 56 pieces.
constexpr int kCostPerTile = 2;
constexpr int kCostPerUnit = 1;

// Tile share of pair `cid`: tiles [lo, hi) of the flat order of all units'
// tiles, where the boundaries split the units' total cost (kCostPerTile per
// tile plus kCostPerUnit per unit with tiles) into equal parts: a tile belongs
// to the pair whose part holds the tile's start.  With a workspace the share
// is exact and the units at its ends may be split with the neighbouring pairs
// (their pieces are merged through the workspace); without one the pair owns
// the whole units whose first tile falls in its share.  Units without tiles (o = 0,
// lse = -inf) are dealt round-robin elsewhere: unit u to pair u mod pairs.
// Both CTAs of a pair compute the same range.  Called by all NT threads of
// the CTA (a multiple of 32, at most 512; at most 256 pairs).
template <int TILE, int NT>
__device__ __forceinline__ void partition_tiles(const PartialParams& pp, int cid, int ncl,
                                                TileRange& rng, Shares& sh, bool& split) {
  static_assert(NT % 32 == 0 && NT <= 512, "block size");
  constexpr int kWarps = NT / 32;
  __shared__ unsigned long long s_scan[kWarps];
  __shared__ int s_load[256];
  __shared__ int s_rng[4];
  __shared__ int s_bound[257];
  // each unit's tile count, written by the thread that owns the unit in the
  // first pass and read back by it in the later ones (a unit lookup is a
  // chain of integer divisions: recomputed in every pass, it made the
  // partition 7 us long at the start of every launch with one unit per
  // thread, 14 us with four)
  constexpr int kNtCache = 2048;
  __shared__ int s_nt[kNtCache];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  sh.total = 0;
  sh.ncl = ncl;
  split = false;
  const int U = pp.num_units;
  const int per = (U + NT - 1) / NT;
  const int a = min(U, static_cast<int>(threadIdx.x) * per);
  const int e = min(U, a + per);
  int cnt = 0, cost = 0;   // tiles and cost of this thread's units
  for (int u = a; u < e; ++u) {
    const int nt = unit_info<TILE>(pp, u).ntiles;
    if (u < kNtCache) s_nt[u] = nt;
    cnt += nt;
    cost += nt > 0 ? kCostPerTile * nt + kCostPerUnit : 0;
  }
  // this thread's own entries only: no barrier needed before reading them
  auto unit_tiles = [&](int u) { return u < kNtCache ? s_nt[u] : unit_info<TILE>(pp, u).ntiles; };
  // exclusive block scan of (cost, tiles), packed in one 64-bit word (both
  // sums stay below 2^32): warp inclusive scans, then the warp totals
  const unsigned long long mine = (static_cast<unsigned long long>(cost) << 32) | static_cast<unsigned>(cnt);
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  if (threadIdx.x == 0) {
    s_rng[0] = INT_MAX;   // u_begin
    s_rng[1] = 0;         // j_begin
    s_rng[2] = -1;        // u_last
    s_rng[3] = 0;         // j_stop
  }
  for (int c = threadIdx.x; c < ncl; c += NT) s_load[c] = 0;
  __syncthreads();
  unsigned long long warp_base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const unsigned long long t = s_scan[w];
    warp_base += w < warp ? t : 0;
    all += t;
  }
  const unsigned long long before = warp_base + incl - mine;
  const int my_start = static_cast<int>(before & 0xffffffffu);      // tiles before this thread's units
  const int64_t my_cstart = static_cast<int64_t>(before >> 32);     // their cost
  const int64_t all_cost = static_cast<int64_t>(all >> 32);
  sh.total = static_cast<int64_t>(all & 0xffffffffu);
  sh.ncl = ncl;
  sh.bound = s_bound;
  // Share boundaries: bound[c] = the tiles whose start lies below the cost
  // target floor(c * cost / ncl).  Every target falls in exactly one unit with
  // tiles (their cost ranges tile [0, cost)), whose thread writes it.
  if (all_cost > 0) {
    int64_t trun = my_start, crun = my_cstart;
    for (int u = a; u < e; ++u) {
      const int nt = unit_tiles(u);
      if (nt == 0) continue;
      const int64_t cend = crun + kCostPerTile * nt + kCostPerUnit;
      for (int c = max(1, static_cast<int>((crun * ncl + all_cost - 1) / all_cost)); c < ncl; ++c) {
        const int64_t tc = static_cast<int64_t>(c) * all_cost / ncl;
        if (tc >= cend) break;
        // tile j of the unit starts at crun + kCostPerUnit + kCostPerTile * j
        const int64_t into = tc - crun - kCostPerUnit;
        const int64_t j = into <= 0 ? 0 : min(static_cast<int64_t>(nt), (into + kCostPerTile - 1) / kCostPerTile);
        s_bound[c] = static_cast<int>(trun + j);
      }
      trun += nt;
      crun = cend;
    }
  } else {
    for (int c = threadIdx.x; c <= ncl; c += NT) s_bound[c] = 0;
  }
  if (threadIdx.x == 0) {
    s_bound[0] = 0;
    s_bound[ncl] = static_cast<int>(sh.total);
  }
  __syncthreads();
  if (pp.split && sh.total > 0) {
    // Split units only where whole units would leave the busiest pair above
    // the even share of cost by more than max(3 tiles, 1/8 of the share): the
    // merge kernel and the extra unit ends cost about that much.
    int64_t run = my_start;
    for (int u = a; u < e; ++u) {
      const int nt = unit_tiles(u);
      if (nt > 0) atomicAdd(&s_load[sh.cluster_of(run)], kCostPerTile * nt + kCostPerUnit);
      run += nt;
    }
    __syncthreads();
    int mx = 0;
    for (int c = threadIdx.x; c < ncl; c += NT) mx = max(mx, s_load[c]);
    const int64_t even = (all_cost + ncl - 1) / ncl;
    // any pair above the threshold decides for all
    split = __syncthreads_or(mx > even + max(int64_t{3 * kCostPerTile}, even / 8)) != 0;
  }
  const int64_t lo = sh.start(cid);
  const int64_t hi = sh.start(cid + 1);
  int64_t run = my_start;
  for (int u = a; u < e; ++u) {
    const int nt = unit_tiles(u);
    if (nt > 0 && lo < hi) {
      if (split) {
        if (lo >= run && lo < run + nt) {
          s_rng[0] = u;
          s_rng[1] = static_cast<int>(lo - run);
        }
        if (hi - 1 >= run && hi - 1 < run + nt) {
          s_rng[2] = u;
          s_rng[3] = static_cast<int>(hi - run);
        }
      } else if (run >= lo && run < hi) {
        atomicMin(&s_rng[0], u);
        atomicMax(&s_rng[2], u);
      }
    }
    run += nt;
  }
  __syncthreads();
  rng.u_begin = s_rng[0];
  rng.j_begin = s_rng[1];
  rng.u_last = s_rng[2];
  // (after the barrier above every thread's entries of s_nt are visible)
  rng.j_stop = split ? s_rng[3]
                     : (rng.u_last < 0 ? 0
                        : rng.u_last < kNtCache ? s_nt[rng.u_last]
                                                : unit_info<TILE>(pp, rng.u_last).ntiles);
  rng.t_begin = static_cast<int>(lo);
  // the unit table of this range (every thread of the CTA passes here)
  const int ncache = rng.u_begin <= rng.u_last ? min(rng.u_last - rng.u_begin + 1, kUnitCache) : 0;
  if (static_cast<int>(threadIdx.x) < ncache)
    s_unit_cache[threadIdx.x] = unit_info<TILE>(pp, rng.u_begin + static_cast<int>(threadIdx.x));
  if (threadIdx.x == 0) {
    s_unit_range[0] = rng.u_begin;
    s_unit_range[1] = ncache;
  }
  __syncthreads();
}

// Record, for the merge kernel, the split unit whose last tile pair `cid`
// holds (if any): the unit at the start of its share, cut before it and
// ending inside it.  Written on every call with a workspace.
template <int TILE>
__device__ __forceinline__ void record_split_unit(const PartialParams& pp, int cid,
                                                  const TileRange& rng, const Shares& sh,
                                                  bool split) {
  int4 rec = make_int4(-1, 0, 0, 0);
  if (split && rng.u_begin <= rng.u_last && rng.j_begin > 0) {
    const int nt = unit_info<TILE>(pp, rng.u_begin).ntiles;
    if (rng.u_begin < rng.u_last || rng.j_stop == nt) {
      const int64_t ustart = sh.start(cid) - rng.j_begin;
      rec = make_int4(rng.u_begin, static_cast<int>(ustart), sh.cluster_of(ustart), cid);
    }
  }
  pp.ws_units[cid] = rec;
  pp.ws_bounds[cid] = static_cast<int>(sh.start(cid));
  if (cid == 0) {
    pp.ws_units[sh.ncl] = make_int4(static_cast<int>(sh.total), sh.ncl, 0, 0);
    pp.ws_bounds[sh.ncl] = static_cast<int>(sh.total);
  }
}

// Protocol waits of the pipelines: each gives up after `limit` polls, records
// MLA_DEV_WAIT_TIMEOUT and raises the CTA's abort flag; a wait that sees the
// flag raised by another warp gives up too.  (The drains at the end of a
// kernel, which wait for copies and MMAs already issued, use mbar_wait with
// the fixed kSpinLimit: those always complete.)
// The polling loops are out of line: a wait that is already satisfied costs
// one try_wait at the call site, and the many call sites of the pipelines do
// not each carry a copy of the loop (the kernels' per-tile code then stays
// small enough for the instruction cache).
static __device__ __noinline__ bool wait_spin_slow(uint64_t* b, uint32_t parity, uint32_t limit,
                                            volatile int* abort_flag, int* err) {
  for (uint32_t it = 0; it < limit; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 1023u) == 1023u && *abort_flag) return false;
  }
  set_error(err, kDevWaitTimeout);
  *abort_flag = 1;
  return false;
}

static __device__ __noinline__ bool wait_lazy_slow(uint64_t* b, uint32_t parity, uint32_t limit,
                                            volatile int* abort_flag, int* err) {
  for (uint32_t it = 0; it < limit; ++it) {
    if (mbar_try_wait_sleep(b, parity, kLazyWaitNs)) return true;
    if ((it & 15u) == 15u && *abort_flag) return false;
  }
  set_error(err, kDevWaitTimeout);
  *abort_flag = 1;
  return false;
}

static __device__ __noinline__ bool wait_cluster_slow(uint64_t* b, uint32_t parity, uint32_t limit,
                                               volatile int* abort_flag, int* err) {
  for (uint32_t it = 0; it < limit; ++it) {
    if (mbar_try_wait_cluster(b, parity)) return true;
    if ((it & 1023u) == 1023u && *abort_flag) return false;
  }
  set_error(err, kDevWaitTimeout);
  *abort_flag = 1;
  return false;
}

struct Waits {
  uint32_t limit;
  volatile int* abort_flag;
  int* err;
  __device__ __forceinline__ bool wait(uint64_t* b, uint32_t parity) const {
    return mbar_try_wait(b, parity) || wait_spin_slow(b, parity, limit, abort_flag, err);
  }
  // waits of whole warp groups off the issue path: polls may suspend
  __device__ __forceinline__ bool lazy(uint64_t* b, uint32_t parity) const {
    return mbar_try_wait(b, parity) || wait_lazy_slow(b, parity, limit, abort_flag, err);
  }
  __device__ __forceinline__ bool cluster(uint64_t* b, uint32_t parity) const {
    return mbar_try_wait_cluster(b, parity) ||
           wait_cluster_slow(b, parity, limit, abort_flag, err);
  }
};

// TMA box `l` (of `br` rows) of the tile of a TileIter.  fetch_id only
// issues the block-table load of the lane's box (one tile ahead); box_row,
// called when that tile is issued, checks the id and forms the row, so a
// producer never waits on a table load.  Boxes past the unit's end re-read
// its last box (in bounds, masked out by the softmax).  Block sizes are
// powers of two (bs_shift = log2 bs).
template <int TILE>
__device__ __forceinline__ int fetch_id(const PartialParams& pp, const TileIter<TILE>& t, int br,
                                        int l, int bs_shift) {
  if (!t.valid || t.ui.current) return 0;
  const int tk = min(t.ui.lo + t.j * TILE + l * br, t.ui.hi - 1);
  return __ldg(pp.block_table + static_cast<int64_t>(t.ui.b) * pp.max_blocks + (tk >> bs_shift));
}

template <int TILE>
__device__ __forceinline__ int box_row(const PartialParams& pp, const TileIter<TILE>& t, int br,
                                       int l, int id, int bs_shift) {
  if (t.ui.current) return t.ui.b * pp.q_len + l * br;
  int tk = t.ui.lo + t.j * TILE + l * br;
  const bool past = tk >= t.ui.hi;
  if (past) tk = t.ui.hi - 1;
  if (id < 0 || id >= pp.num_blocks) {
    set_error(pp.err, kDevBadBlockId);
    id = 0;
  }
  int row = (id << bs_shift) + (tk & (pp.bs - 1));
  if (past) row &= ~(br - 1);
  return row;
}

// Merge of the units split across pairs (launched after a partial kernel
// that had a workspace; programmatic dependent launch).
int launch_partial_merge(const PartialParams& pp, int clusters, cudaStream_t stream);

}  // namespace mla
