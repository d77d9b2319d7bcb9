// Partial attention per context shard: mla_dcp_decode_partial.
//
// One decode step of MLA reads a paged latent KV cache.  Each cached token is
// a 512-wide latent c_KV plus a 64-wide RoPE key k_R (MLA multi-GPU TP
// article, "物理矛盾").  The history is split along the sequence into shards;
// each shard (and the causal CURRENT chunk) yields a partial output and its
// log-sum-exp (vllm-ascend PR #16977 study page: glossary "DCP", "LSE"; the
// HISTORY and CURRENT attention calls of code blocks B and C).
//
// Work unit = (sequence b, query token i, part p).  Per unit, with the 128
// query heads of token i as the M dimension of every MMA:
//   S = Q . K^T        Q [128 x 576], K = tile of 128 cached tokens x 576
//   P = exp2(S*scale*log2e - m)   online softmax (running max m, lazy rescale)
//   O += P . V         V = the same tokens' latent columns, [128 x 512]
//
// GB300 mapping: a SPLIT-ROLE PAIR of CTAs (a 2-CTA cluster on two SMs).
// A 128 x 512 fp32 accumulator fills one SM's whole tensor memory, and
// tensor-core MMAs only run at full rate with N >= 128, so the work is split
// by role rather than by data:
//   rank 0 ("QK CTA"): Q's latent part lives in its TMEM (the A operand of
//     tcgen05 MMAs straight from tensor memory), the RoPE part in SMEM;
//     S = Q K^T for 128-token tiles (N = 128) into two TMEM buffers; online
//     softmax; P (bf16/fp16) plus per-row rescale factor, row sum and running
//     max are shipped to rank 1 with one shared-memory-to-shared-memory bulk
//     copy per tile (DSMEM, 256 B per token, one direction).
//   rank 1 ("PV CTA"): the full fp32 O [128 x 512] in its TMEM; O += P V with
//     N = 256 MMAs; rescale of O when the running max moved; epilogue O / l
//     and the LSE.
// Each CTA TMA-loads the KV columns it needs (rank 0 all 576, rank 1 the 512
// latent ones, close in time so the second read hits L2).
//
// Scheduling: a persistent grid of every co-resident pair.  The units' tiles
// form one flat sequence that the pairs share either as whole units or, with
// a workspace and when whole units would be uneven, as exact tile shares; a
// unit cut between pairs leaves pieces (O / l and LSE) in the workspace that
// mla_partial_merge_kernel combines afterwards.
//
// Warp roles (256 threads per CTA):
//   rank 0: w0 TMA producer (K chunks + Q RoPE), w1 MMA issuer, w2-3 LSE of
//           empty parts, w4-7 softmax + Q latent loader (thread = head row)
//   rank 1: w0 TMA producer (V), w1 MMA issuer, w2 hands P buffers back,
//           w3 zeros of empty parts, w4-7 O rescale + epilogue (thread = row)
// Every wait is bounded; on timeout the kernel records MLA_DEV_WAIT_TIMEOUT,
// raises an abort flag, drains its own copies and MMAs, frees TMEM, returns.
#include <mutex>
#include "partial_sched.cuh"

namespace mla {

// Shared-memory plan (offsets from a 1024-aligned base; same size on both
// ranks).  Rank 0: K ring, Q RoPE tile, one outgoing P message.
// Rank 1: V ring, two incoming P messages, the epilogue's staging rows.
// Barriers at one common offset.
//
// A ring stage is one mbarrier phase.  Each phase costs an SM a fixed few
// hundred nanoseconds however many bytes it carries (measured on GB300: a
// TMA stream with 8 KB per phase reaches 25 GB/s per SM, with 64 KB per
// phase the full HBM rate from half the SMs), so the K ring moves three
// 64-dim chunks (48 KB) per phase: a 128-token tile is exactly 3 stages.
struct PairSmem {
  static constexpr int kTile = 128;
  static constexpr int kKChunk = kTile * 128;          // one 64-dim chunk of a tile
  static constexpr int kKPer = 3;                      // chunks per K stage
  static constexpr int kKStage = kKPer * kKChunk;      // 48 KB
  static constexpr int kNK = 3;                        // K stages: one tile
  static constexpr int kQStages = (8 + kKPer - 1) / kKPer;   // stages of a query's 8 latent chunks
  static constexpr int kVSub = 64;                     // tokens per V stage
  static constexpr int kVChunk = kVSub * 128;          // one 64-dim chunk of a V stage
  static constexpr int kVStage = 8 * kVChunk;          // 64 tokens x 512 latent (64 KB)
  static constexpr int kNV = 2;
  // P message: P [128 rows x 128 tokens] as two 64-token SW128 chunks,
  // alpha[128], lsum[128], header.
  static constexpr int kMsgP = 2 * 16384;
  static constexpr int kMsgAlpha = kMsgP;
  static constexpr int kMsgL = kMsgAlpha + 512;
  static constexpr int kMsgM = kMsgL + 512;
  static constexpr int kMsgHdr = kMsgM + 512;
  static constexpr int kMsgBytes = kMsgHdr + 16;       // 34320, multiple of 16
  static constexpr int kMsgStride = 34816;             // 1024-aligned slot
  // rank 0
  static constexpr int kKOff = 0;
  static constexpr int kQrOff = kKOff + kNK * kKStage;       // 147456
  static constexpr int kPsOff = kQrOff + 16384;              // 163840 (one outgoing message)
  static constexpr int kEnd0 = kPsOff + kMsgStride;          // 198656
  // rank 1
  static constexpr int kVOff = 0;
  static constexpr int kPrOff = kVOff + kNV * kVStage;       // 131072
  static constexpr int kStgOff = kPrOff + 2 * kMsgStride;    // 200704: 4 KB per epilogue warp
  static constexpr int kEnd1 = kStgOff + 4 * 4096;           // 217088
  static constexpr int kBarOff = kEnd0 > kEnd1 ? kEnd0 : kEnd1;
  static constexpr int kTotal = kBarOff + 512 + 1024;
};
static_assert(9 == PairSmem::kNK * PairSmem::kKPer, "a tile's 9 chunks fill the K ring's stages exactly");
static_assert(PairSmem::kTotal <= 232448, "shared memory budget");

// Barrier slots in the common block.
// (derived from the ring sizes, so a deeper ring cannot make slots overlap)
enum : int {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + PairSmem::kNK,
  B_QR_FULL = B_KEMPTY + PairSmem::kNK,
  B_Q_EMPTY = B_QR_FULL + 1,
  B_QLAT_FULL = B_Q_EMPTY + 1,
  B_S_FULL = B_QLAT_FULL + 1,      // 2
  B_S_EMPTY = B_S_FULL + 2,        // 2
  B_PFREE = B_S_EMPTY + 2,         // 2
  B_MMA_DONE_A = B_PFREE + 2,
  B_VFULL = B_MMA_DONE_A + 1,
  B_VEMPTY = B_VFULL + PairSmem::kNV,
  B_P_FULL = B_VEMPTY + PairSmem::kNV,   // 2
  B_PV_DONE = B_P_FULL + 2,        // 2
  B_META_READ = B_PV_DONE + 2,     // 2
  B_O_EMPTY = B_META_READ + 2,
  B_O_FIXED = B_O_EMPTY + 1,
  B_MMA_DONE_B = B_O_FIXED + 1,
  B_MSG_FREE = B_MMA_DONE_B + 1,   // rank 0: the outgoing P message has landed in rank 1
  B_COUNT = B_MSG_FREE + 1
};
// barriers + TMEM slot + abort flag + 4 warp flags + Q-stage counters + the
// P message count must fit the barrier block
static_assert((B_COUNT + 9) * 8 <= 512, "barrier block");

// Epilogue of one piece, rows of this warp: row r (TMEM lane r) of O times
// `mul`, in the partial dtype, to `dst_row` (this thread's output row, or
// nullptr for a row that is not stored).  Per 128-byte column chunk, each
// lane writes its row into the warp's 4 KB of staging (16-byte unit j of row
// r at unit j ^ (r & 7), so neither the row writes nor the read-back below
// conflict on banks), then the warp stores the chunk back four rows per
// instruction: each store covers whole 128-byte row segments instead of one
// 32-byte piece of 32 different rows.  The warp's O_EMPTY arrival comes after
// its last store is issued: released as soon as the last TMEM load had landed,
// the next unit's PV MMAs ran against the staging traffic and the very long
// context was 1 % slower.
__device__ __forceinline__ void epilogue_rows(uint32_t ta, uint32_t stg, char* dst_row, float mul,
                                              int dt, int lane, uint64_t* o_empty) {
  const bool f32 = dt == kFP32;
  const int nchunk = f32 ? 16 : 8;
  for (int c = 0; c < nchunk; ++c) {
    uint32_t w[32];
    if (f32) {
      uint32_t v[32];
      tmem_ld32(ta + c * 32, v);
      tmem_wait_ld(v);
#pragma unroll
      for (int t = 0; t < 32; ++t) w[t] = __float_as_uint(__uint_as_float(v[t]) * mul);
    } else {
      uint32_t v0[32], v1[32];
      tmem_ld32(ta + c * 64, v0);
      tmem_ld32(ta + c * 64 + 32, v1);
      tmem_wait_ld(v0, v1);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        w[k] = pack2_dt(__uint_as_float(v0[2 * k]) * mul, __uint_as_float(v0[2 * k + 1]) * mul, dt);
        w[16 + k] =
            pack2_dt(__uint_as_float(v1[2 * k]) * mul, __uint_as_float(v1[2 * k + 1]) * mul, dt);
      }
    }
    __syncwarp();   // the read-back of the previous chunk is done
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                   w[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 4 + (lane >> 3), j = lane & 7;
      char* d = reinterpret_cast<char*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst_row), rr));
      const uint4 x = ld_shared_v4(stg + rr * 128 + ((j ^ (rr & 7)) << 4));
      if (d != nullptr) *reinterpret_cast<uint4*>(d + c * 128 + j * 16) = x;
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(o_empty);
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                       const __grid_constant__ CUtensorMap tm_qpe,
                       const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_cur,
                       const __grid_constant__ CUtensorMap tm_kv_v,
                       const __grid_constant__ CUtensorMap tm_cur_v, const PartialParams pp) {
  using L = PairSmem;
  constexpr int TILE = L::kTile;
  constexpr int kTmemCols = 512;
  constexpr uint32_t kQlatCol = 0;       // rank 0: Q latent, 256 packed columns
  constexpr uint32_t kSCol = 256;        // rank 0: S buffers [256,384), [384,512)
  constexpr float kRescaleThresh = 8.0f; // lazy rescale: only when max grows by > 2^8

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + B_COUNT + 1);
  volatile uint32_t* warp_flags = reinterpret_cast<volatile uint32_t*>(bar + B_COUNT + 2);
  int* q_readers = reinterpret_cast<int*>(bar + B_COUNT + 4);   // warps done with Q stage
  // rank 0: P messages sent; rank 1: P messages the PV issuer has seen land
  volatile int* msg_count = reinterpret_cast<volatile int*>(bar + B_COUNT + 8);

  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = pp.err;

  if (threadIdx.x == 0) {
    if (rank == 0) {
      for (int s = 0; s < L::kNK; ++s) {
        mbar_init(&bar[B_KFULL + s], 1);
        mbar_init(&bar[B_KEMPTY + s], 1);
      }
      mbar_init(&bar[B_QR_FULL], 1);
      mbar_init(&bar[B_Q_EMPTY], 1);
      mbar_init(&bar[B_QLAT_FULL], 4);
      for (int k = 0; k < 2; ++k) {
        mbar_init(&bar[B_S_FULL + k], 1);
        mbar_init(&bar[B_S_EMPTY + k], 4);
        mbar_init(&bar[B_PFREE + k], 1);
      }
      mbar_init(&bar[B_MMA_DONE_A], 1);
      mbar_init(&bar[B_MSG_FREE], 1);
      for (int c = 0; c < PairSmem::kQStages; ++c) q_readers[c] = 0;
    } else {
      for (int s = 0; s < L::kNV; ++s) {
        mbar_init(&bar[B_VFULL + s], 1);
        mbar_init(&bar[B_VEMPTY + s], 1);
      }
      for (int k = 0; k < 2; ++k) {
        mbar_init(&bar[B_P_FULL + k], 1);
        mbar_init(&bar[B_PV_DONE + k], 1);
        mbar_init(&bar[B_META_READ + k], 4);
      }
      mbar_init(&bar[B_O_EMPTY], 4);
      mbar_init(&bar[B_O_FIXED], 4);
      mbar_init(&bar[B_MMA_DONE_B], 1);
      // the first two P messages may land as soon as the cluster is up
      mbar_arrive_expect_tx(&bar[B_P_FULL + 0], L::kMsgBytes);
      mbar_arrive_expect_tx(&bar[B_P_FULL + 1], L::kMsgBytes);
    }
    *abort_flag = 0;
    *msg_count = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_qlat);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_kv);
    prefetch_tmap(&tm_cur);
    prefetch_tmap(&tm_kv_v);
    prefetch_tmap(&tm_cur_v);
  }
  __syncthreads();
  cluster_sync();   // every barrier of both CTAs is initialised
  griddep_launch_dependents();   // a dependent merge grid may be scheduled as CTAs retire
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Tile share of this pair (partition_tiles); units without tiles are
  // dealt round-robin: unit u to pair u mod pairs, so a batch of short or
  // empty histories spreads its zero rows over every pair.
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(nclusters_x());
  TileRange rng;
  Shares shares;
  bool split = false;
  partition_tiles<TILE, 256>(pp, cid, ncl, rng, shares, split);

  const Waits waits{pp.spin_limit, abort_flag, err};
  auto wait = [&](uint64_t* b, uint32_t parity) { return waits.wait(b, parity); };
  auto wait_lazy = [&](uint64_t* b, uint32_t parity) { return waits.lazy(b, parity); };
  auto wait_cl = [&](uint64_t* b, uint32_t parity) { return waits.cluster(b, parity); };
  const int bs_shift = __ffs(pp.bs) - 1;   // block sizes are powers of two
  auto fetch_id = [&](const TileIter<TILE>& t, int br, int l) {
    return mla::fetch_id<TILE>(pp, t, br, l, bs_shift);
  };
  auto box_row = [&](const TileIter<TILE>& t, int br, int l, int id) {
    return mla::box_row<TILE>(pp, t, br, l, id, bs_shift);
  };
  const int br_k = pp.box_rows;           // rank 0 box rows: min(128, bs)
  const int br_v = pp.box_rows_v;         // rank 1 box rows: min(32, bs)

  if (rank == 0) {
    uint8_t* sK = smem + L::kKOff;
    uint8_t* sQr = smem + L::kQrOff;
    uint8_t* sPs = smem + L::kPsOff;
    if (warp == 0) {
      // ------------------------------------------------ rank 0: TMA producer
      // The whole warp runs the loop converged: every lane polls the stage
      // barrier and lane l issues box l of each chunk (no shuffles, no
      // divergent single-lane sections on the issue path).
      TileIter<TILE> it;
      it.start(pp, rng);
      int cs = 0;
      int qloads = 0;
      bool ok = true;
      const int nbox = TILE / br_k;      // boxes per chunk of a tile (1, 2 or 8)
      const bool boxlane = lane < nbox;
      int id_cur = boxlane ? fetch_id(it, br_k, lane) : 0;
      while (it.valid) {
        const UnitInfo ui = it.ui;
        TileIter<TILE> nx = it;
        nx.advance(pp);
        const int id_next = boxlane ? fetch_id(nx, br_k, lane) : 0;
        if (it.first() && it.newq) {
          const int qrow = (ui.b * pp.q_len + ui.i) * pp.H;
          // Q latent of the new query: eight 64-column chunks through the
          // ring (3 + 3 + 2 per stage), ahead of the unit's K (the softmax
          // warps move them to TMEM)
          for (int qs = 0; qs < L::kQStages; ++qs) {
            const int st = cs % L::kNK;
            if (cs >= L::kNK && !wait(&bar[B_KEMPTY + st], ((cs / L::kNK) - 1) & 1)) {
              ok = false;
              break;
            }
            const int nc = min(L::kKPer, 8 - qs * L::kKPer);
            if (lane == 0) {
              mbar_arrive_expect_tx(&bar[B_KFULL + st], nc * L::kKChunk);
              for (int k = 0; k < nc; ++k)
                tma_load_2d(sK + st * L::kKStage + k * L::kKChunk, &tm_qlat, &bar[B_KFULL + st],
                            (qs * L::kKPer + k) * 64, qrow);
            }
            ++cs;
          }
          if (!ok) break;
          // Q RoPE tile: its buffer is free once the previous query's MMAs are done
          if (it.nq >= 1 && !wait(&bar[B_Q_EMPTY], (it.nq - 1) & 1)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar[B_QR_FULL], 16384);
            tma_load_2d(sQr, &tm_qpe, &bar[B_QR_FULL], 0, qrow);
          }
          ++qloads;
        }
        // (after the Q loads: the box rows wait for the block-table entries)
        const int row = boxlane ? box_row(it, br_k, lane, id_cur) : 0;
        const CUtensorMap* map = ui.current ? &tm_cur : &tm_kv;
        uint8_t* dst = sK + lane * br_k * 128;
        for (int ks = 0; ks < L::kNK; ++ks) {
          const int st = cs % L::kNK;
          if (cs >= L::kNK && !wait(&bar[B_KEMPTY + st], ((cs / L::kNK) - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar[B_KFULL + st], L::kKStage);
          if (boxlane) {
#pragma unroll
            for (int k = 0; k < L::kKPer; ++k) {
              const int c = ks * L::kKPer + k;
              tma_load_2d(dst + st * L::kKStage + k * L::kKChunk, map, &bar[B_KFULL + st], c * 64,
                          row);
            }
          }
          ++cs;
        }
        if (!ok) break;
        id_cur = id_next;
        it = nx;
      }
      if (lane == 0) {
        // drain: the last chunk issued into each stage has landed
        for (int s = 0; s < L::kNK && s < cs; ++s) {
          const int last = cs - 1 - ((cs - 1 - s) % L::kNK);
          mbar_wait(&bar[B_KFULL + s], (last / L::kNK) & 1, err);
        }
        if (qloads > 0) mbar_wait(&bar[B_QR_FULL], (qloads - 1) & 1, err);
      }
    } else if (warp == 1) {
      // ------------------------------------------------ rank 0: MMA issuer (QK)
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc_f16(128, TILE, BF16, false, false);
        const uint32_t k_base = smem_u32(sK);
        const uint32_t qr_base = smem_u32(sQr);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0, cs = 0;
        bool ok = true;
        while (ok && it.valid) {
          if (it.first() && it.newq) {
            if (!wait(&bar[B_QLAT_FULL], it.nq & 1) || !wait(&bar[B_QR_FULL], it.nq & 1)) {
              ok = false;
              break;
            }
            cs += L::kQStages;   // the Q latent stages in the ring are the softmax warps' to free
          }
          const int sb = g & 1;
          if (g >= 2 && !wait(&bar[B_S_EMPTY + sb], ((g >> 1) - 1) & 1)) { ok = false; break; }
          const uint32_t d = tmem + kSCol + sb * TILE;
          for (int ks = 0; ks < L::kNK; ++ks) {
            const int st = cs % L::kNK;
            if (!wait(&bar[B_KFULL + st], (cs / L::kNK) & 1)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < L::kKPer; ++k) {
              const int c = ks * L::kKPer + k;
              const uint32_t kb = k_base + st * L::kKStage + k * L::kKChunk;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = make_desc_sw128(kb + kk * 32, 16, 1024);
                if (c < 8)
                  umma_ts(d, tmem + kQlatCol + c * 32 + kk * 8, bd, idesc, (c | kk) ? 1u : 0u);
                else
                  umma_ss(d, make_desc_sw128(qr_base + kk * 32, 16, 1024), bd, idesc, 1u);
              }
            }
            umma_commit(&bar[B_KEMPTY + st]);
            ++cs;
          }
          if (!ok) break;
          umma_commit(&bar[B_S_FULL + sb]);
          if (it.last_of_q(pp)) umma_commit(&bar[B_Q_EMPTY]);
          it.advance(pp);
          ++g;
        }
        umma_commit(&bar[B_MMA_DONE_A]);
        mbar_wait(&bar[B_MMA_DONE_A], 0, err);
      }
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------ rank 0: LSE of empty parts
      const int t = threadIdx.x - 64;
      for (int u = cid; u < pp.num_units; u += ncl) {
        const UnitInfo ui = unit_info<TILE>(pp, u);
        if (ui.ntiles != 0) continue;
        const int64_t tok = static_cast<int64_t>(ui.b) * pp.q_len + ui.i;
        for (int h = t; h < pp.H; h += 64) pp.lse_part[part_row(pp, tok, ui.p, h)] = -INFINITY;
      }
    } else {
      // ------------------------------------------------ rank 0: softmax
      const int r = threadIdx.x - 128;           // TMEM lane == head row
      const int wq = warp & 3;
      const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t precv_peer = map_to_peer(smem + L::kPrOff, 1);
      const uint32_t pfull_peer = map_to_peer(&bar[B_P_FULL], 1);
      TileIter<TILE> it;
      it.start(pp, rng);
      int g = 0;
      int cq = 0;   // ring position in stages: kQStages per new query, kNK per tile
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      while (ok && it.valid) {
        const UnitInfo ui = it.ui;
        if (it.first()) {
          if (it.newq) {
            // Q latent row r -> TMEM (packed pairs, low half = even element),
            // from the eight ring stages the producer filled for this query
            // (the softmax warps meet at named barriers, so every exit
            // decision is made together through named_bar_and)
            const bool qe = it.nq < 1 || wait_lazy(&bar[B_Q_EMPTY], (it.nq - 1) & 1);
            if (!named_bar_and(1, 128, qe)) { ok = false; break; }
            tc_fence_after();
            // each warp copies its 32 rows of a chunk; the last warp done
            // with a stage frees it (no block-wide barrier per stage)
            for (int c = 0; c < 8; ++c) {
              const int qs = c / L::kKPer, k = c % L::kKPer;
              const int st = (cq + qs) % L::kNK;
              if (k == 0 && !wait_lazy(&bar[B_KFULL + st], ((cq + qs) / L::kNK) & 1)) {
                ok = false;
                break;
              }
              // row r of a 128-byte-swizzled chunk: 16-byte unit j at (j ^ (r & 7))
              const uint8_t* rowp = sK + st * L::kKStage + k * L::kKChunk + r * 128;
              uint32_t w[32];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint4 x = *reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4));
                if (r >= pp.H) x = make_uint4(0, 0, 0, 0);   // rows of the next query
                w[4 * j] = x.x;
                w[4 * j + 1] = x.y;
                w[4 * j + 2] = x.z;
                w[4 * j + 3] = x.w;
              }
              tmem_st32(tmem + lane_base + kQlatCol + c * 32, w);   // consumes the loads
              if (k == L::kKPer - 1 || c == 7) {
                __syncwarp();
                if (lane == 0) {
                  __threadfence_block();
                  if (atomicAdd(&q_readers[qs], 1) == 3) {
                    q_readers[qs] = 0;
                    mbar_arrive(&bar[B_KEMPTY + st]);
                  }
                }
              }
            }
            cq += L::kQStages;
            if (!named_bar_and(1, 128, ok)) { ok = false; break; }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_QLAT_FULL]);
          }
          m = -INFINITY;
          l = 0.f;
        }
        const int sb = g & 1;
        if (!named_bar_and(1, 128, wait_lazy(&bar[B_S_FULL + sb], (g >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[TILE];
        // S in four 32-column loads, one at a time, each folded into the row
        // max before the next is issued: register-bound TMEM reads slow the
        // SM's TMA stream, and they do so least when they are not bursts
        const int nvalid = min(TILE, ui.hi - (ui.lo + it.j * TILE));
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        {
          const uint32_t sa = tmem + lane_base + kSCol + sb * TILE;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(sa + 32 * c, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              const int tt = 32 * c + t;
              s[tt] = tt < nvalid ? __uint_as_float(v[t]) * pp.scale_log2 : -INFINITY;
              mx[t & 3] = fmaxf(mx[t & 3], s[tt]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_S_EMPTY + sb]);

        // ---- online softmax in the log2 domain
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        bool need_rescale = false;
        float alpha = 1.f;
        if (it.first()) {
          m = mt;
        } else if (mt > m + kRescaleThresh) {
          need_rescale = true;
          alpha = fast_exp2(m - mt);
          m = mt;
        }
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < TILE; ++t) {
          s[t] = fast_exp2(s[t] - m);     // masked: exp2(-inf) = 0
          ps[t & 3] += s[t];
        }
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));

        // ---- P message for rank 1
        // Single outgoing buffer: the copy of tile g-1 has finished reading
        // it once that message has landed in rank 1, which rank 1 reports on
        // B_MSG_FREE (a shared-to-cluster bulk copy completes only on the
        // destination's mbarrier; no wait of the sender tracks it).
        uint8_t* msg = sPs;
        bool mfree = true;
        if (threadIdx.x == 128 && g >= 1) mfree = wait_cl(&bar[B_MSG_FREE], (g - 1) & 1);
        if (!named_bar_and(1, 128, mfree)) { ok = false; break; }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            const int t = half * 64 + uu * 8;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack2<BF16>(s[t + 2 * e], s[t + 2 * e + 1]);
            *reinterpret_cast<uint4*>(msg + half * 16384 + sw128_offset(r, uu)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        reinterpret_cast<float*>(msg + L::kMsgAlpha)[r] = alpha;
        reinterpret_cast<float*>(msg + L::kMsgL)[r] = l;
        reinterpret_cast<float*>(msg + L::kMsgM)[r] = m;
        const uint32_t any = __any_sync(0xffffffffu, need_rescale) ? 1u : 0u;
        if (lane == 0) warp_flags[wq] = any;
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (threadIdx.x == 128) {
          const uint32_t flags = (warp_flags[0] | warp_flags[1] | warp_flags[2] | warp_flags[3]) |
                                 (it.last() ? 2u : 0u);
          *reinterpret_cast<volatile uint32_t*>(msg + L::kMsgHdr) = flags;
          fence_proxy_async_smem();
          if (g >= 2 && !wait_cl(&bar[B_PFREE + sb], ((g >> 1) - 1) & 1)) ok = false;
          if (ok) {
            bulk_copy_to_peer(precv_peer + sb * L::kMsgStride, msg, L::kMsgBytes,
                              pfull_peer + sb * 8);
            *msg_count = g + 1;
          }
        }
        ok = named_bar_and(1, 128, ok && !*abort_flag);
        it.advance(pp);
        ++g;
        cq += L::kNK;
      }
    }
  } else {
    uint8_t* sV = smem + L::kVOff;
    uint8_t* sPr = smem + L::kPrOff;
    if (warp == 0) {
      // ------------------------------------------------ rank 1: TMA producer (V)
      // Converged warp: lane (bb * 8 + c) issues latent chunk c of box bb of
      // each 32-token stage; lanes 0..nbox-1 hold the tile's box rows.
      TileIter<TILE> it;
      it.start(pp, rng);
      int vs = 0;
      bool ok = true;
      const int nbox = TILE / br_v;           // boxes per tile (4 or 8)
      const int sub_boxes = L::kVSub / br_v;  // boxes per 32-token stage (1 or 2)
      const int vc = lane & 7, vb = lane >> 3;
      const bool vlane = vb < sub_boxes;
      const bool boxlane = lane < nbox;
      int id_cur = boxlane ? fetch_id(it, br_v, lane) : 0;
      while (it.valid) {
        const UnitInfo ui = it.ui;
        TileIter<TILE> nx = it;
        nx.advance(pp);
        const int id_next = boxlane ? fetch_id(nx, br_v, lane) : 0;
        const int my_row = boxlane ? box_row(it, br_v, lane, id_cur) : 0;
        const CUtensorMap* map = ui.current ? &tm_cur_v : &tm_kv_v;
        uint8_t* dst = sV + vc * L::kVChunk + vb * br_v * 128;
        for (int sub = 0; sub < TILE / L::kVSub; ++sub) {
          const int st = vs % L::kNV;
          const int row = __shfl_sync(0xffffffffu, my_row, (sub * sub_boxes + vb) & 7);
          if (vs >= L::kNV && !wait(&bar[B_VEMPTY + st], ((vs / L::kNV) - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar[B_VFULL + st], L::kVStage);
          if (vlane)
            tma_load_2d(dst + st * L::kVStage, map, &bar[B_VFULL + st], vc * 64, row);
          ++vs;
        }
        if (!ok) break;
        id_cur = id_next;
        it = nx;
      }
      if (lane == 0)
        for (int s = 0; s < L::kNV && s < vs; ++s) {
          const int last = vs - 1 - ((vs - 1 - s) % L::kNV);
          mbar_wait(&bar[B_VFULL + s], (last / L::kNV) & 1, err);
        }
    } else if (warp == 1) {
      // ------------------------------------------------ rank 1: MMA issuer (PV)
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc_f16(128, 256, BF16, false, true);
        const uint32_t v_base = smem_u32(sV);
        const uint32_t p_base = smem_u32(sPr);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0, vs = 0, nfix = 0;
        bool ok = true;
        while (ok && it.valid) {
          const int sb = g & 1;
          if (!wait(&bar[B_P_FULL + sb], (g >> 1) & 1)) { ok = false; break; }
          const uint32_t hdr =
              *reinterpret_cast<volatile uint32_t*>(sPr + sb * L::kMsgStride + L::kMsgHdr);
          const bool first = it.first();
          if (first && it.k >= 1 && !wait(&bar[B_O_EMPTY], (it.k - 1) & 1)) { ok = false; break; }
          if (hdr & 1u) {
            if (!wait(&bar[B_O_FIXED], nfix & 1)) { ok = false; break; }
            ++nfix;
          }
          const uint32_t pa = p_base + sb * L::kMsgStride;
          for (int sub = 0; sub < TILE / L::kVSub; ++sub) {
            const int st = vs % L::kNV;
            if (!wait(&bar[B_VFULL + st], (vs / L::kNV) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t vb = v_base + st * L::kVStage;
#pragma unroll
            for (int kk = 0; kk < L::kVSub / 16; ++kk) {
              const int tok = sub * L::kVSub + kk * 16;
              const uint64_t ad = make_desc_sw128(pa + (tok >> 6) * 16384 + (tok & 63) * 2, 16, 1024);
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint64_t bd =
                    make_desc_sw128(vb + half * 4 * L::kVChunk + kk * 2048, L::kVChunk, 1024);
                umma_ss(tmem + half * 256, ad, bd, idesc, (first && sub == 0 && kk == 0) ? 0u : 1u);
              }
            }
            umma_commit(&bar[B_VEMPTY + st]);
            ++vs;
          }
          if (!ok) break;
          umma_commit(&bar[B_PV_DONE + sb]);
          it.advance(pp);
          ++g;
        }
        umma_commit(&bar[B_MMA_DONE_B]);
        mbar_wait(&bar[B_MMA_DONE_B], 0, err);
      }
    } else if (warp == 2) {
      // ------------------------------------------------ rank 1: hand P buffers back
      if (lane == 0) {
        const uint32_t pfree_peer = map_to_peer(&bar[B_PFREE], 0);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0;
        while (it.valid) {
          const int sb = g & 1;
          if (!wait(&bar[B_PV_DONE + sb], (g >> 1) & 1)) break;
          if (!wait(&bar[B_META_READ + sb], (g >> 1) & 1)) break;
          mbar_arrive_expect_tx(&bar[B_P_FULL + sb], L::kMsgBytes);   // tile g + 2
          mbar_arrive_remote(pfree_peer + sb * 8);
          it.advance(pp);
          ++g;
        }
      }
    } else if (warp == 3) {
      // ------------------------------------------------ rank 1: zeros of empty parts
      for (int u = cid; u < pp.num_units; u += ncl) {
        const UnitInfo ui = unit_info<TILE>(pp, u);
        if (ui.ntiles != 0) continue;
        const int64_t tok = static_cast<int64_t>(ui.b) * pp.q_len + ui.i;
        for (int h = 0; h < pp.H; ++h) {
          const int64_t e0 = part_row(pp, tok, ui.p, h) * 512;
          if (pp.part_dtype == kFP32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(pp.o_part) + e0);
            for (int c = lane; c < 128; c += 32) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(pp.o_part) + e0);
            for (int c = lane; c < 64; c += 32) o[c] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // ------------------------------------------------ rank 1: P landing watcher
      // Reports each P message to rank 0 as soon as it has landed (the
      // sender's single buffer is then free) and counts them for the drain
      // at the end of the kernel.  A message lands only in an armed slot,
      // and rank 0 sends message g + 2 only after this report for g + 1, so
      // the watcher can never fall a whole phase behind on a slot.
      if (lane == 0) {
        const uint32_t msgfree_peer = map_to_peer(&bar[B_MSG_FREE], 0);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0;
        while (it.valid) {
          if (!wait(&bar[B_P_FULL + (g & 1)], (g >> 1) & 1)) break;
          *msg_count = g + 1;
          mbar_arrive_remote(msgfree_peer);
          it.advance(pp);
          ++g;
        }
      }
    } else {
      // ------------------------------------------------ rank 1: O rescale + epilogue
      const int r = threadIdx.x - 128;
      const int wq = warp & 3;
      const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t stg = smem_u32(smem + L::kStgOff + wq * 4096);
      TileIter<TILE> it;
      it.start(pp, rng);
      int g = 0;
      bool ok = true;
      while (ok && it.valid) {
        const UnitInfo ui = it.ui;
        const int sb = g & 1;
        if (!wait_lazy(&bar[B_P_FULL + sb], (g >> 1) & 1)) { ok = false; break; }
        const uint8_t* msg = sPr + sb * L::kMsgStride;
        const uint32_t hdr = *reinterpret_cast<const volatile uint32_t*>(msg + L::kMsgHdr);
        const float alpha = reinterpret_cast<const float*>(msg + L::kMsgAlpha)[r];
        const float lsum = reinterpret_cast<const float*>(msg + L::kMsgL)[r];
        const float m2 = reinterpret_cast<const float*>(msg + L::kMsgM)[r];
        // the message's header fields are in registers: the slot may go back
        // (once the PV MMAs have read its P as well)
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_META_READ + sb]);
        if (hdr & 1u) {
          // O *= alpha before PV of this tile; PV of the previous tile must be done
          if (!wait_lazy(&bar[B_PV_DONE + ((g - 1) & 1)], ((g - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          for (int c0 = 0; c0 < 512; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + c0, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
            tmem_st32(tmem + lane_base + c0, v);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[B_O_FIXED]);
        }
        if (hdr & 2u) {
          // epilogue of the piece: O / l and its LSE
          if (!wait_lazy(&bar[B_PV_DONE + sb], (g >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const float lse2 = m2 + __log2f(lsum);          // log2 domain
          const int64_t row_out =
              part_row(pp, static_cast<int64_t>(ui.b) * pp.q_len + ui.i, ui.p, r);   // r < H only
          const float inv_l = 1.f / lsum;
          const int64_t row_bytes = pp.part_dtype == kFP32 ? 2048 : 1024;
          // A piece of a unit split across pairs parks O / l (in the partial
          // dtype) and the LSE in this pair's workspace slot instead; the
          // pieces are merged after the main loop (rows < H only).
          const bool whole = it.whole();
          const int slot = 2 * cid + (it.u == rng.u_begin ? 0 : 1);
          char* dst = nullptr;
          if (r < pp.H)
            dst = whole ? static_cast<char*>(pp.o_part) + row_out * row_bytes
                        : static_cast<char*>(pp.ws_o) + (static_cast<int64_t>(slot) * 128 + r) * row_bytes;
          epilogue_rows(tmem + lane_base, stg, dst, inv_l, pp.part_dtype, lane, &bar[B_O_EMPTY]);
          if (!whole)
            pp.ws_lse[slot * 128 + r] = lse2;
          else if (r < pp.H)
            pp.lse_part[row_out] = lse2 * kLn2;
        }
        it.advance(pp);
        ++g;
      }
    }
  }

  // every tensor-memory access of this thread has completed (a warp that left
  // the Q copy early may still have stores in flight) before TMEM is freed
  __syncwarp();
  tmem_wait_st();
  tmem_wait_ld();
  tc_fence_before();
  __syncthreads();
  if (pp.split && rank == 1 && threadIdx.x == 0) record_split_unit<TILE>(pp, cid, rng, shares, split);
  cluster_sync();
  if (rank == 1 && threadIdx.x == 64) {
    // Drain the P messages rank 0 sent that the PV issuer never saw land
    // (it stops early when a wait runs out): rank 0 must not exit while its
    // copies still read its buffer, nor rank 1 while they still write here.
    // Every message went to an armed slot, so each completes a P_FULL phase.
    const uint32_t sent_addr = map_to_peer(const_cast<int*>(msg_count), 0);
    int sent;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sent) : "r"(sent_addr) : "memory");
    for (int k = *msg_count; k < sent; ++k) mbar_wait(&bar[B_P_FULL + (k & 1)], (k >> 1) & 1, err);
  }
  cluster_sync();   // no DSMEM traffic into either CTA after this point
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- merge of split units
// One CTA per (pair, 32-row quarter): merges the pieces of the split unit
// whose last tile that pair held (pp.ws_units[pair]) by their LSEs, exactly as
// the combine merges shards, and writes the unit's o_part rows and lse_part.
// Eight threads per row, 64 columns each; every thread folds the pieces in
// pair order into a running (max, weight sum, accumulator) of its own, so the
// CTA needs no shared memory and no barrier, and a launch takes few dependent
// memory round trips (record, share boundaries, then each piece's LSE and
// values together).
__global__ void __launch_bounds__(256, 2) mla_partial_merge_kernel(PartialParams pp) {
  griddep_wait();   // the partial grid has completed and its writes are visible
  griddep_launch_dependents();
  const int4 rec = pp.ws_units[blockIdx.x];
  const int u = rec.x;
  const int r = blockIdx.y * 32 + (threadIdx.x >> 3);
  if (u < 0 || r >= pp.H) return;
  const int64_t ustart = rec.y;
  const int c_first = rec.z, c_last = rec.w;
  const int sub = threadIdx.x & 7;      // 64-column slice of the row
  const bool f32 = pp.part_dtype == kFP32;
  float acc[64];
#pragma unroll
  for (int t = 0; t < 64; ++t) acc[t] = 0.f;
  float m = -INFINITY, wsum = 0.f;
  for (int c = c_first; c <= c_last; ++c) {
    const int s0 = pp.ws_bounds[c], s1 = pp.ws_bounds[c + 1];
    if (s1 <= s0) continue;                               // pair without tiles
    const int sl = 2 * c + (s0 >= ustart ? 0 : 1);        // its first or its last piece
    const float l = pp.ws_lse[sl * 128 + r];              // log2 domain
    const int64_t e0 = (static_cast<int64_t>(sl) * 128 + r) * 512 + sub * 64;
    if (l > m) {   // a new reference maximum (the first piece: the scale is 0)
      const float sc = exp2f(m - l);
#pragma unroll
      for (int t = 0; t < 64; ++t) acc[t] *= sc;
      wsum *= sc;
      m = l;
    }
    const float w = exp2f(l - m);
    wsum += w;
    // the piece's 64 values in two halves (fewer live registers: two CTAs
    // per SM, so every CTA of a launch is resident at once)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float x[32];
      if (f32) {
        const float4* src =
            reinterpret_cast<const float4*>(static_cast<const float*>(pp.ws_o) + e0 + 32 * half);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 f = src[q];
          x[4 * q] = f.x;
          x[4 * q + 1] = f.y;
          x[4 * q + 2] = f.z;
          x[4 * q + 3] = f.w;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(pp.ws_o) +
                                                          e0 + 32 * half);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 h = src[q];
          const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f2 = unpack2(hw[j], pp.part_dtype);
            x[8 * q + 2 * j] = f2.x;
            x[8 * q + 2 * j + 1] = f2.y;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) acc[32 * half + t] = fmaf(w, x[t], acc[32 * half + t]);
    }
  }
  const float inv = 1.f / wsum;
  const int ib = u / pp.P;
  const int64_t row = part_row(pp, static_cast<int64_t>(ib % pp.B) * pp.q_len + ib / pp.B, u % pp.P, r);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(acc[32 * h + t]);
    store_row32(pp.o_part, row * 512 + sub * 64 + 32 * h, v, inv, pp.part_dtype);
  }
  if (sub == 0) pp.lse_part[row] = (m + __log2f(wsum)) * kLn2;
}

// ---------------------------------------------------------------- launcher
// Sets the kernel's shared-memory limit and finds how many CTA pairs fit on
// the current device at once (cached per device).
// The cache is keyed by device ordinal and guarded by a lock, so host threads
// that make their first call at the same time set it up once.  A device reset
// (cudaDeviceReset) does not clear it; the occupancy it holds stays valid for
// the same GPU.
template <bool BF16>
static int prepare_partial(int* clusters) {
  static int cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    auto kern = mla_partial_kernel<BF16>;
    constexpr int smem = PairSmem::kTotal;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int mc = 0;
    if (cudaOccupancyMaxActiveClusters(&mc, kern, &cfg) != cudaSuccess || mc < 1) return -1;
    cache[dev] = std::min(mc, 256);   // the partition keeps per-pair state in 256-entry arrays
  }
  *clusters = cache[dev];
  return 0;
}

// Pairs that every partial kernel (16-bit and E4M3 caches) can hold at once:
// the workspace is sized for this many.
int partial_max_clusters() {
  int a = 0, b = 0;
  if (prepare_partial<true>(&a) != 0 || prepare_partial<false>(&b) != 0) return -1;
  const int c = partial_fp8_max_clusters();
  if (c < 1) return -1;
  return std::min(std::min(a, b), c);
}

template <bool BF16>
static int launch_partial_t(const CUtensorMap& qlat, const CUtensorMap& qpe, const CUtensorMap& kv,
                            const CUtensorMap& cur, const CUtensorMap& kv_v,
                            const CUtensorMap& cur_v, const PartialParams& pp,
                            cudaStream_t stream) {
  int max_clusters = 0;
  if (prepare_partial<BF16>(&max_clusters) != 0) return -1;
  // with a workspace every resident pair takes a share (equal shares of cost)
  const int clusters = pp.split ? pp.split : std::max(1, std::min(pp.num_units, max_clusters));
  if (clusters > max_clusters) return -1;
  mla_partial_kernel<BF16><<<dim3(2 * clusters), dim3(256), PairSmem::kTotal, stream>>>(
      qlat, qpe, kv, cur, kv_v, cur_v, pp);
  return pp.split ? launch_partial_merge(pp, clusters, stream) : 0;
}

// Programmatic dependent launch: the merge grid is scheduled while the
// partial grid drains and waits for it on the device (griddepcontrol).
int launch_partial_merge(const PartialParams& pp, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters, 4, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_partial_merge_kernel, pp) != cudaSuccess ? -1 : 0;
}

int launch_partial(const CUtensorMap& qlat, const CUtensorMap& qpe, const CUtensorMap& kv,
                   const CUtensorMap& cur, const CUtensorMap& kv_v, const CUtensorMap& cur_v,
                   const PartialParams& pp, bool bf16, cudaStream_t stream) {
  return bf16 ? launch_partial_t<true>(qlat, qpe, kv, cur, kv_v, cur_v, pp, stream)
              : launch_partial_t<false>(qlat, qpe, kv, cur, kv_v, cur_v, pp, stream);
}

}  // namespace mla
