// Partial attention per context shard over an FP8 (E4M3) latent cache:
// mla_dcp_decode_partial_fp8.
//
// Every cached value (latent c_KV and RoPE key k_R, history and CURRENT) is
// one E4M3 byte times a per-tensor kv_scale; the attention is the one of the
// 16-bit kernel (partial.cu) on those values.  The work units, the tile
// shares of the CTA pairs, the split-role pair and its P-message protocol are
// the same; what changes is how each CTA feeds its tensor cores:
//
//   rank 0 (QK CTA): a K tile is 128 tokens x 576 bytes, moved by TMA as five
//     128-byte chunks (four latent, one RoPE chunk whose upper 64 bytes are the
//     zero fill of an out-of-range box) straight into kind::f8f6f4 MMAs
//     (E4M3 x E4M3, fp32 accumulate).  The 16-bit query row is turned into
//     E4M3 once per query token with a power-of-two row scale sq and two
//     terms, q = sq * (hi + lo) + e with hi = rn(q / sq), lo = rn(q / sq - hi):
//     |e| <= 2^-8 |q| + 2^-17 max|q_row|, about the precision of bf16.  S is
//     accumulated as Q_hi K^T + Q_lo K^T (two MMAs per k-step: the tensor
//     work of the 16-bit kernel, on half the bytes).
//   rank 1 (PV CTA): O += P V as kind::f8f6f4 MMAs straight on the E4M3 V
//     bytes that TMA lands (V as the MN-major B operand: latent-contiguous
//     token rows, as the cache stores them), with P in the same two-term
//     form: p' = 2^6 p (p <= 2^2 under the lazy-rescale threshold, so
//     p' <= 256 and the bulk of p' lies in E4M3's normal range),
//     hi = rn(p'), lo = rn(p' - hi).  Rank 0 sends p' in fp16 (its exp2 and
//     the fp16 packing are the softmax's whole conversion work); rank 1's
//     epilogue warps split it into the two E4M3 terms in place, so the
//     conversion work of a tile is shared by the two SMs.
// kv_scale is folded into the softmax scale and into the epilogue's 1 / l
// (l is the row sum of p', so the 2^6 cancels).
//
// Warp roles (384 threads per CTA; two 4-warp groups per row set, group
// A = w4-7, group B = w8-11, thread = TMEM lane = head row):
//   rank 0: w0 TMA producer (query chunks, K tiles), w1 MMA issuer, w2-3 LSE
//           of empty parts; group A quantises each new query, then both
//           groups run the softmax of a tile, A on its columns 0..63 and B
//           on 64..127 (the row max is exchanged through shared memory)
//   rank 1: w0 TMA producer (E4M3 V), w1 MMA issuer, w2 hands P buffers
//           back, w3 zeros of empty parts; groups A / B
//           rescale O and write the epilogue of latent columns 0..255 /
//           256..511
// Every wait is bounded, as in the 16-bit kernel.
#include <cuda_fp8.h>
#include <mutex>
#include "partial_sched.cuh"

namespace mla {

namespace {

// Shared-memory plan (offsets from a 1024-aligned base; same size on both ranks).
struct Fp8Smem {
  static constexpr int kTile = 128;
  static constexpr int kChunk = kTile * 128;         // 128 rows x 128 bytes (16 KB)
  static constexpr int kKPer = 5;                    // chunks per K stage: 4 latent + RoPE
  static constexpr int kKStage = kKPer * kChunk;     // 80 KB: one tile per ring phase
  static constexpr int kNK = 2;
  static constexpr int kQStages = 2;                 // a query's 9 16-bit chunks: 5 + 4
  static constexpr int kV8Sub = 64;                  // tokens per E4M3 V stage
  static constexpr int kV8Chunk = kV8Sub * 128;      // 128 latent bytes x 64 tokens (8 KB)
  static constexpr int kV8Stage = 4 * kV8Chunk;      // 32 KB
  static constexpr int kNV8 = 4;
  // P message: P' [128 rows x 128 tokens] fp16 as two 64-token 128-byte-
  // swizzled 16 KB tiles (rewritten in place by rank 1 as [hi | lo] E4M3
  // bytes of the same 64 tokens per 128-byte row), alpha[128], the row sums
  // of the two column halves lA[128] and lB[128], m[128], header.
  static constexpr int kMsgP = 2 * 16384;
  static constexpr int kMsgAlpha = kMsgP;
  static constexpr int kMsgLA = kMsgAlpha + 512;
  static constexpr int kMsgLB = kMsgLA + 512;
  static constexpr int kMsgM = kMsgLB + 512;
  static constexpr int kMsgHdr = kMsgM + 512;
  static constexpr int kMsgBytes = kMsgHdr + 16;     // 34832, multiple of 16
  static constexpr int kMsgStride = 35840;           // 1024-aligned slot
  // rank 0
  static constexpr int kKOff = 0;
  static constexpr int kQr8Off = kKOff + kNK * kKStage;   // 163840: query RoPE, hi | lo bytes
  static constexpr int kEnd0 = kQr8Off + 16384;           // 180224
  // (rank 0 has no message buffer: its softmax threads write each P message
  // straight into rank 1's landing slot with st.async)
  // rank 1
  static constexpr int kV8Off = 0;
  static constexpr int kPrOff = kV8Off + kNV8 * kV8Stage;      // 131072
  static constexpr int kEnd1 = kPrOff + 2 * kMsgStride;        // 202752
  static constexpr int kBarOff = kEnd0 > kEnd1 ? kEnd0 : kEnd1;
  static constexpr int kTotal = kBarOff + 512 + 1024;
};
static_assert(Fp8Smem::kTotal <= 232448, "shared memory budget");
static_assert(Fp8Smem::kTile == 2 * Fp8Smem::kV8Sub, "a tile is two E4M3 V stages");

enum : int {
  F_KFULL = 0,
  F_KEMPTY = F_KFULL + Fp8Smem::kNK,
  F_Q_EMPTY = F_KEMPTY + Fp8Smem::kNK,
  F_QLAT_FULL = F_Q_EMPTY + 1,
  F_S_FULL = F_QLAT_FULL + 1,     // 2
  F_S_EMPTY = F_S_FULL + 2,       // 2
  F_PFREE = F_S_EMPTY + 2,        // 2
  F_MMA_DONE_A = F_PFREE + 2,
  F_V8FULL = F_MMA_DONE_A + 1,
  F_V8EMPTY = F_V8FULL + Fp8Smem::kNV8,
  F_P_FULL = F_V8EMPTY + Fp8Smem::kNV8,     // 2
  F_PV_DONE = F_P_FULL + 2,       // 2
  F_META_READ = F_PV_DONE + 2,    // 2
  F_O_EMPTY = F_META_READ + 2,
  F_O_FIXED = F_O_EMPTY + 1,
  F_MMA_DONE_B = F_O_FIXED + 1,
  F_P8_READY = F_MMA_DONE_B + 1,  // 2: a landed P' is in its E4M3 form
  F_COUNT = F_P8_READY + 2
};
// barriers + TMEM slot + abort flag + 4 warp flags + the P message count
static_assert((F_COUNT + 9) * 8 <= 512, "barrier block");

// Two floats -> two E4M3 bytes (round to nearest even, saturating at 448),
// a in the low byte.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// P' = 2^kPShift p: the lazy-rescale threshold keeps p <= 2^kRescaleThresh,
// so p' <= 2^8 (inside E4M3's 448).
constexpr float kRescaleThresh = 2.0f;
constexpr int kPShift = 8 - 2;


// Two fp16 p' values -> their E4M3 hi bytes and lo bytes (low element in the
// low byte of each): hi = rn(p'), lo = rn(p' - hi); the remainder is exact in
// fp16 (p' and hi share a binade, hi has 4 significant bits).
__device__ __forceinline__ void split_e4m3x2(uint32_t p2, uint32_t& hi, uint32_t& lo) {
  __half2_raw pr;
  pr.x = static_cast<unsigned short>(p2 & 0xFFFFu);
  pr.y = static_cast<unsigned short>(p2 >> 16);
  hi = __nv_cvt_halfraw2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(hi), __NV_E4M3);
  const __half2 rem = __hsub2(*reinterpret_cast<const __half2*>(&pr), *reinterpret_cast<const __half2*>(&hr));
  lo = __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&rem), __NV_SATFINITE, __NV_E4M3);
}

// Two E4M3 bytes (the low one first) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t v) {
  const uint32_t h = e4m3x2_to_f16x2(v);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Eight 16-bit query values (one 16-byte unit), times inv_sq, as the two
// E4M3 terms: hi[0..1] and lo[0..1] each hold 8 bytes in element order.
template <bool BF16>
__device__ __forceinline__ void quantize8(uint4 x, float inv_sq, uint32_t (&hi)[2],
                                          uint32_t (&lo)[2]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t h16[4], l16[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = unpack2(w[k], BF16 ? kBF16 : kFP16);
    const float a = f.x * inv_sq, b = f.y * inv_sq;
    h16[k] = to_e4m3x2(a, b);
    const float2 d = e4m3x2_to_float2(h16[k]);
    l16[k] = to_e4m3x2(a - d.x, b - d.y);
  }
  hi[0] = h16[0] | (h16[1] << 16);
  hi[1] = h16[2] | (h16[3] << 16);
  lo[0] = l16[0] | (l16[1] << 16);
  lo[1] = l16[2] | (l16[3] << 16);
}

template <bool BF16>
__device__ __forceinline__ float amax8(uint4 x, float m) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = unpack2(w[k], BF16 ? kBF16 : kFP16);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

// Query row r of a new query token -> its two E4M3 terms: the latent part
// into TMEM (hi at column t_hi, lo at t_lo, 4 bytes per column), the RoPE
// part into row r of the 128-byte-swizzled sQr tile (hi bytes in units 0..3,
// lo bytes in units 4..7).  The row's 16-bit chunks (8 latent, then RoPE)
// are chunks 0..4 of ring stage st0 and 0..3 of st1.  Returns the row's
// score factor scale_log2 * sq.  Out of line: it runs once per query token,
// and the softmax loop it belongs to stays small.
template <bool BF16>
__device__ __noinline__ float quantize_query_row(const uint8_t* st0, const uint8_t* st1, int r,
                                                 bool live, uint32_t t_hi, uint32_t t_lo,
                                                 uint8_t* sQr, float scale_log2) {
  auto qrow_ptr = [&](int c) -> const uint8_t* {
    return (c < 5 ? st0 + c * Fp8Smem::kChunk : st1 + (c - 5) * Fp8Smem::kChunk) + r * 128;
  };
  float amax = 0.f;
  for (int c = 0; c < 9; ++c) {
    const uint8_t* rowp = qrow_ptr(c);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      amax = amax8<BF16>(*reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4)), amax);
  }
  if (!live) amax = 0.f;
  // row scale sq = 2^(E - 8) with amax = f * 2^E, f in [0.5, 1): the row's
  // largest value maps into [128, 256)
  int E = 0;
  frexpf(amax, &E);
  const float inv_sq = live && amax > 0.f ? ldexpf(1.f, 8 - E) : 0.f;
  for (int c = 0; c < 9; ++c) {
    const uint8_t* rowp = qrow_ptr(c);
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t h2[2], l2[2];
      quantize8<BF16>(*reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4)), inv_sq, h2, l2);
      hi[2 * j] = h2[0];
      hi[2 * j + 1] = h2[1];
      lo[2 * j] = l2[0];
      lo[2 * j + 1] = l2[1];
    }
    if (c < 8) {
      // 64 values = 16 columns of 4 bytes
      tmem_st16(t_hi + c * 16, hi);
      tmem_st16(t_lo + c * 16, lo);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        *reinterpret_cast<uint4*>(sQr + sw128_offset(r, u)) =
            make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
        *reinterpret_cast<uint4*>(sQr + sw128_offset(r, 4 + u)) =
            make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
      }
    }
  }
  return scale_log2 * (amax > 0.f ? ldexpf(1.f, E - 8) : 1.f);
}

// O *= alpha on columns [cbeg, cbeg + NC) of this thread's TMEM row.
// (This and store_o_half stay inline: as out-of-line functions called from
// more than one site, their warp-collective TMEM loads returned zeros in one
// template instance.)
template <int NC>
__device__ __forceinline__ void rescale_o(uint32_t trow, int cbeg, float alpha) {
  for (int c0 = cbeg; c0 < cbeg + NC; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(trow + c0, v);
    tmem_wait_ld(v);
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
    tmem_st32(trow + c0, v);
  }
  tmem_wait_st();
}

// Columns [cbeg, cbeg + NC) of this thread's TMEM row, times mul, stored as
// NC values of dtype dt at element e0 + cbeg of dst.
template <int NC>
__device__ __forceinline__ void store_o_half(uint32_t trow, int cbeg, void* dst, int64_t e0, float mul,
                                          int dt, bool active) {
  for (int c0 = cbeg; c0 < cbeg + NC; c0 += 64) {
    uint32_t v0[32], v1[32];
    tmem_ld32(trow + c0, v0);
    tmem_ld32(trow + c0 + 32, v1);
    tmem_wait_ld(v0, v1);
    if (active) {
      store_row32(dst, e0 + c0, v0, mul, dt);
      store_row32(dst, e0 + c0 + 32, v1, mul, dt);
    }
  }
}

}  // namespace

// Warp groups (4 warps each) that share a tile's softmax on rank 0 (by
// columns) and O's rescale / epilogue on rank 1 (by latent columns).
constexpr int kGroups = 2;
constexpr int kFp8Threads = 128 + 128 * kGroups;
constexpr int kSCols = 128 / kGroups;    // S columns (tokens) per softmax thread
constexpr int kOCols = 512 / kGroups;    // O columns per epilogue thread

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFp8Threads, 1)
    mla_partial_fp8_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                           const __grid_constant__ CUtensorMap tm_qpe,
                           const __grid_constant__ CUtensorMap tm_kv,
                           const __grid_constant__ CUtensorMap tm_cur,
                           const __grid_constant__ CUtensorMap tm_kv_v,
                           const __grid_constant__ CUtensorMap tm_cur_v, const PartialParams pp) {
  using L = Fp8Smem;
  constexpr int TILE = L::kTile;
  constexpr int kTmemCols = 512;
  constexpr uint32_t kQhiCol = 0;        // rank 0: query hi bytes, 128 columns (4 per column)
  constexpr uint32_t kQloCol = 128;      // rank 0: query lo bytes, 128 columns
  constexpr uint32_t kSCol = 256;        // rank 0: S buffers [256,384), [384,512)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + F_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + F_COUNT + 1);
  volatile uint32_t* warp_flags = reinterpret_cast<volatile uint32_t*>(bar + F_COUNT + 2);
  // rank 0: the softmax groups' row maxima of a tile and group A's row factors
  __shared__ float s_rowmax[kGroups][128];
  __shared__ float s_fs[128];
  // rank 0: P messages sent; rank 1: P messages the watcher has seen land
  volatile int* msg_count = reinterpret_cast<volatile int*>(bar + F_COUNT + 8);

  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = pp.err;

  if (threadIdx.x == 0) {
    if (rank == 0) {
      for (int s = 0; s < L::kNK; ++s) {
        mbar_init(&bar[F_KFULL + s], 1);
        mbar_init(&bar[F_KEMPTY + s], 1);
      }
      mbar_init(&bar[F_Q_EMPTY], 1);
      mbar_init(&bar[F_QLAT_FULL], 4);
      for (int k = 0; k < 2; ++k) {
        mbar_init(&bar[F_S_FULL + k], 1);
        mbar_init(&bar[F_S_EMPTY + k], 4 * kGroups);
        mbar_init(&bar[F_PFREE + k], 1);
      }
      mbar_init(&bar[F_MMA_DONE_A], 1);
    } else {
      for (int s = 0; s < L::kNV8; ++s) {
        mbar_init(&bar[F_V8FULL + s], 1);
        mbar_init(&bar[F_V8EMPTY + s], 1);
      }
      for (int k = 0; k < 2; ++k) {
        mbar_init(&bar[F_P_FULL + k], 1);
        mbar_init(&bar[F_PV_DONE + k], 1);
        mbar_init(&bar[F_META_READ + k], 4 * kGroups);
      }
      mbar_init(&bar[F_O_EMPTY], 4 * kGroups);
      mbar_init(&bar[F_O_FIXED], 4 * kGroups);
      mbar_init(&bar[F_MMA_DONE_B], 1);
      mbar_init(&bar[F_P8_READY + 0], 4 * kGroups);
      mbar_init(&bar[F_P8_READY + 1], 4 * kGroups);
      // the first two P messages may land as soon as the cluster is up
      mbar_arrive_expect_tx(&bar[F_P_FULL + 0], L::kMsgBytes);
      mbar_arrive_expect_tx(&bar[F_P_FULL + 1], L::kMsgBytes);
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

  // Tile share of this pair (partition_tiles); units without tiles are dealt
  // round-robin: unit u to pair u mod pairs.
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(nclusters_x());
  TileRange rng;
  Shares shares;
  bool split = false;
  partition_tiles<TILE, kFp8Threads>(pp, cid, ncl, rng, shares, split);

  const Waits waits{pp.spin_limit, abort_flag, err};
  auto wait = [&](uint64_t* b, uint32_t parity) { return waits.wait(b, parity); };
  auto wait_lazy = [&](uint64_t* b, uint32_t parity) { return waits.lazy(b, parity); };
  auto wait_cl = [&](uint64_t* b, uint32_t parity) { return waits.cluster(b, parity); };
  const int bs_shift = __ffs(pp.bs) - 1;   // block sizes are powers of two
  const int br_k = pp.box_rows;            // rank 0 box rows: min(128, bs)
  const int br_v = pp.box_rows_v;          // rank 1 box rows: min(64, bs)

  if (rank == 0) {
    uint8_t* sK = smem + L::kKOff;
    uint8_t* sQr = smem + L::kQr8Off;
    if (warp == 0) {
      // ------------------------------------------------ rank 0: TMA producer
      // Converged warp: every lane polls the stage barrier, lane l issues box
      // l of each chunk of a tile.
      TileIter<TILE> it;
      it.start(pp, rng);
      int cs = 0;
      bool ok = true;
      const int nbox = TILE / br_k;      // boxes per chunk of a tile (1, 2, 4 or 8)
      const bool boxlane = lane < nbox;
      int id_cur = boxlane ? fetch_id<TILE>(pp, it, br_k, lane, bs_shift) : 0;
      while (it.valid) {
        const UnitInfo ui = it.ui;
        TileIter<TILE> nx = it;
        nx.advance(pp);
        const int id_next = boxlane ? fetch_id<TILE>(pp, nx, br_k, lane, bs_shift) : 0;
        if (it.first() && it.newq) {
          // the new query's eight 64-column latent chunks and its RoPE chunk
          // (16-bit) through the ring, 5 + 4 per stage; the softmax warps
          // turn them into E4M3 terms
          const int qrow = (ui.b * pp.q_len + ui.i) * pp.H;
          for (int qs = 0; qs < L::kQStages; ++qs) {
            const int st = cs % L::kNK;
            if (cs >= L::kNK && !wait(&bar[F_KEMPTY + st], ((cs / L::kNK) - 1) & 1)) {
              ok = false;
              break;
            }
            const int nc = qs == 0 ? 5 : 4;
            if (lane == 0) {
              mbar_arrive_expect_tx(&bar[F_KFULL + st], nc * L::kChunk);
              for (int k = 0; k < nc; ++k) {
                const int c = qs * 5 + k;
                uint8_t* dst = sK + st * L::kKStage + k * L::kChunk;
                if (c < 8)
                  tma_load_2d(dst, &tm_qlat, &bar[F_KFULL + st], c * 64, qrow);
                else
                  tma_load_2d(dst, &tm_qpe, &bar[F_KFULL + st], 0, qrow);
              }
            }
            ++cs;
          }
          if (!ok) break;
        }
        // K tile: five 128-byte chunks (bytes [128c, 128c + 128) of each
        // token; chunk 4 reads bytes 512..639 of 576-byte rows, the part past
        // the row is zero-filled)
        const int row = boxlane ? box_row<TILE>(pp, it, br_k, lane, id_cur, bs_shift) : 0;
        const CUtensorMap* map = ui.current ? &tm_cur : &tm_kv;
        const int st = cs % L::kNK;
        if (cs >= L::kNK && !wait(&bar[F_KEMPTY + st], ((cs / L::kNK) - 1) & 1)) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar[F_KFULL + st], L::kKStage);
        if (boxlane) {
          uint8_t* dst = sK + st * L::kKStage + lane * br_k * 128;
#pragma unroll
          for (int c = 0; c < L::kKPer; ++c)
            tma_load_2d(dst + c * L::kChunk, map, &bar[F_KFULL + st], c * 128, row);
        }
        ++cs;
        id_cur = id_next;
        it = nx;
      }
      if (lane == 0) {
        // drain: the last load issued into each stage has landed
        for (int s = 0; s < L::kNK && s < cs; ++s) {
          const int last = cs - 1 - ((cs - 1 - s) % L::kNK);
          mbar_wait(&bar[F_KFULL + s], (last / L::kNK) & 1, err);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------ rank 0: MMA issuer (QK)
      if (lane == 0) {
        // E4M3 x E4M3 -> fp32: format fields 0, both operands K-major
        constexpr uint32_t idesc = make_idesc_f16(128, TILE, false, false, false);
        const uint32_t k_base = smem_u32(sK);
        const uint32_t qr_base = smem_u32(sQr);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0, cs = 0;
        bool ok = true;
        while (ok && it.valid) {
          if (it.first() && it.newq) {
            if (!wait(&bar[F_QLAT_FULL], it.nq & 1)) break;
            cs += L::kQStages;   // the query's ring stages are the softmax warps' to free
          }
          const int sb = g & 1;
          if (g >= 2 && !wait(&bar[F_S_EMPTY + sb], ((g >> 1) - 1) & 1)) break;
          const uint32_t d = tmem + kSCol + sb * TILE;
          const int st = cs % L::kNK;
          if (!wait(&bar[F_KFULL + st], (cs / L::kNK) & 1)) break;
          tc_fence_after();
          const uint32_t kb = k_base + st * L::kKStage;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = make_desc_sw128(kb + c * L::kChunk + kk * 32, 16, 1024);
              umma_ts_f8(d, tmem + kQhiCol + c * 32 + kk * 8, bd, idesc, (c | kk) ? 1u : 0u);
              umma_ts_f8(d, tmem + kQloCol + c * 32 + kk * 8, bd, idesc, 1u);
            }
          }
          // RoPE: 64 bytes per row (two k-steps); the query's hi bytes are
          // bytes 0..63 of its row, the lo bytes 64..127
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t bd = make_desc_sw128(kb + 4 * L::kChunk + kk * 32, 16, 1024);
            umma_ss_f8(d, make_desc_sw128(qr_base + kk * 32, 16, 1024), bd, idesc, 1u);
            umma_ss_f8(d, make_desc_sw128(qr_base + 64 + kk * 32, 16, 1024), bd, idesc, 1u);
          }
          umma_commit(&bar[F_KEMPTY + st]);
          ++cs;
          umma_commit(&bar[F_S_FULL + sb]);
          if (it.last_of_q(pp)) umma_commit(&bar[F_Q_EMPTY]);
          it.advance(pp);
          ++g;
        }
        umma_commit(&bar[F_MMA_DONE_A]);
        mbar_wait(&bar[F_MMA_DONE_A], 0, err);
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
      // ------------------------------------------------ rank 0: query terms + softmax
      // Group A (w4-7) alone turns each new query into its E4M3 terms (named
      // barrier 2); both groups (named barrier 1, 256 threads) then share the
      // tiles' softmax by columns.  Every exit decision is made together
      // through named_bar_and.
      const int grp = (warp - 4) >> 2;
      const int r = (threadIdx.x - 128) & 127;   // TMEM lane == head row
      const int wq = warp & 3;
      const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t precv_peer = map_to_peer(smem + L::kPrOff, 1);
      const uint32_t pfull_peer = map_to_peer(&bar[F_P_FULL], 1);
      TileIter<TILE> it;
      it.start(pp, rng);
      int g = 0;
      int cq = 0;   // ring position in stages: kQStages per new query, one per tile
      float m = -INFINITY, l = 0.f;
      float fs = 0.f;   // this row's score factor: scale * log2(e) * kv_scale * sq
      bool ok = true;
      while (ok && it.valid) {
        const UnitInfo ui = it.ui;
        bool qok = true;
        if (it.first()) {
          if (it.newq && grp == 0) {
            const bool qe = it.nq < 1 || wait_lazy(&bar[F_Q_EMPTY], (it.nq - 1) & 1);
            const bool q0 = qe && wait_lazy(&bar[F_KFULL + cq % L::kNK], (cq / L::kNK) & 1);
            const bool q1 =
                q0 && wait_lazy(&bar[F_KFULL + (cq + 1) % L::kNK], ((cq + 1) / L::kNK) & 1);
            qok = named_bar_and(2, 128, q1);
          }
          if (it.newq && grp == 0 && qok) {
            tc_fence_after();
            // (rows past H hold the next query's rows: zero terms)
            fs = quantize_query_row<BF16>(sK + (cq % L::kNK) * L::kKStage,
                                          sK + ((cq + 1) % L::kNK) * L::kKStage, r, r < pp.H,
                                          tmem + lane_base + kQhiCol, tmem + lane_base + kQloCol,
                                          sQr, pp.scale_log2);
            s_fs[r] = fs;   // group B's copy, read after the next joint barrier
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(2, 128);   // every row has read the query's ring stages
            if (threadIdx.x == 128) {
              mbar_arrive(&bar[F_KEMPTY + cq % L::kNK]);
              mbar_arrive(&bar[F_KEMPTY + (cq + 1) % L::kNK]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[F_QLAT_FULL]);
          }
          if (it.newq) cq += L::kQStages;
          m = -INFINITY;
          l = 0.f;
        }
        const int sb = g & 1;
        if (!named_bar_and(1, 128 * kGroups, qok && wait_lazy(&bar[F_S_FULL + sb], (g >> 1) & 1))) {
          ok = false;
          break;
        }
        if (kGroups > 1 && it.first() && it.newq && grp == 1) fs = s_fs[r];
        tc_fence_after();
        // this group's columns [c0, c0 + kSCols) of the tile, read from TMEM
        // 32 at a time, each folded into the row max before the next is
        // issued; then the S buffer goes back to the MMA
        const int c0 = kSCols * grp;
        const int nvalid = min(TILE, ui.hi - (ui.lo + it.j * TILE)) - c0;
        const uint32_t sa = tmem + lane_base + kSCol + sb * TILE + c0;
        float v[kSCols];
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kSCols / 32; ++c) {
          uint32_t w[32];
          tmem_ld32(sa + 32 * c, w);
          tmem_wait_ld(w);
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            v[32 * c + t] = __uint_as_float(w[t]);
            if (32 * c + t < nvalid) mx[t & 3] = fmaxf(mx[t & 3], v[32 * c + t]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[F_S_EMPTY + sb]);
        const float my_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        if (kGroups > 1) s_rowmax[grp][r] = my_max;
        // rank 1's landing slot sb is free again once the PV MMAs of tile
        // g - 2 have read it (F_PFREE); the barrier also exchanges the maxima
        bool sfree = true;
        if (threadIdx.x == 128 && g >= 2) sfree = wait_cl(&bar[F_PFREE + sb], ((g >> 1) - 1) & 1);
        if (!named_bar_and(1, 128 * kGroups, sfree)) { ok = false; break; }
        float row_max = my_max;
        if (kGroups > 1)
#pragma unroll
          for (int k = 0; k < kGroups; ++k) row_max = fmaxf(row_max, s_rowmax[k][r]);
        const float mt = row_max * fs;   // fs > 0

        // ---- online softmax in the log2 domain
        bool need_rescale = false;
        float alpha = 1.f;
        if (it.first()) {
          m = mt;
        } else if (mt > m + kRescaleThresh) {
          need_rescale = true;
          alpha = fast_exp2(m - mt);
          m = mt;
        }

        // ---- P message, written into rank 1's slot sb with st.async (each
        // store completes its bytes on rank 1's F_P_FULL[sb]): p' = 2^6
        // exp2(s - m) in fp16, this group's 64 tokens = its 16 KB tile
        const uint32_t rmsg = precv_peer + sb * L::kMsgStride;
        const uint32_t rbar = pfull_peer + sb * 8;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        const float mp = static_cast<float>(kPShift) - m;
        // all of p first (independent exp2s), then the packed stores
#pragma unroll
        for (int t = 0; t < kSCols; ++t) {
          // masked columns: 0; others p' <= 2^8
          v[t] = t < nvalid ? fast_exp2(fmaf(v[t], fs, mp)) : 0.f;
          ps[t & 3] += v[t];
        }
#pragma unroll
        for (int uu = 0; uu < kSCols / 8; ++uu) {
          const float* p = v + 8 * uu;
          // 64 tokens per 16 KB tile of the message, 8 per 16-byte unit
          const int tok = c0 + 8 * uu;
          st_async_v4(rmsg + (tok >> 6) * 16384 + sw128_offset(r, (tok & 63) >> 3),
                      make_uint4(pack2<false>(p[0], p[1]), pack2<false>(p[2], p[3]),
                                 pack2<false>(p[4], p[5]), pack2<false>(p[6], p[7])),
                      rbar);
        }
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));   // this group's half of the row sum of p'
        if (grp == 0) {
          st_async_b32(rmsg + L::kMsgAlpha + 4 * r, __float_as_uint(alpha), rbar);
          st_async_b32(rmsg + L::kMsgLA + 4 * r, __float_as_uint(l), rbar);
          st_async_b32(rmsg + L::kMsgM + 4 * r, __float_as_uint(m), rbar);
          // (both groups take the same rescale decisions: group A's flags)
          const uint32_t any = __any_sync(0xffffffffu, need_rescale) ? 1u : 0u;
          if (lane == 0) warp_flags[wq] = any;
          if (kGroups == 1) st_async_b32(rmsg + L::kMsgLB + 4 * r, 0u, rbar);
        } else {
          st_async_b32(rmsg + L::kMsgLB + 4 * r, __float_as_uint(l), rbar);
        }
        named_bar_sync(1, 128 * kGroups);   // every store of the message is issued
        if (threadIdx.x == 128) {
          const uint32_t flags = (warp_flags[0] | warp_flags[1] | warp_flags[2] | warp_flags[3]) |
                                 (it.last() ? 2u : 0u);
          st_async_v4(rmsg + L::kMsgHdr, make_uint4(flags, 0u, 0u, 0u), rbar);
          *msg_count = g + 1;   // messages sent (for rank 1's drain)
        }
        ok = named_bar_and(1, 128 * kGroups, ok && !*abort_flag);
        it.advance(pp);
        ++g;
        cq += 1;
      }
    }
  } else {
    uint8_t* sV8 = smem + L::kV8Off;
    uint8_t* sPr = smem + L::kPrOff;
    if (warp == 0) {
      // ------------------------------------------------ rank 1: TMA producer (E4M3 V)
      // Converged warp: lane (bb * 4 + c) issues 128-byte latent chunk c of
      // box bb of each 64-token stage; lanes 0..nbox-1 hold the tile's box rows.
      TileIter<TILE> it;
      it.start(pp, rng);
      int vs = 0;
      bool ok = true;
      const int nbox = TILE / br_v;            // boxes per tile (2, 4 or 8)
      const int sub_boxes = L::kV8Sub / br_v;  // boxes per 64-token stage (1, 2 or 4)
      const int vc = lane & 3, vb = lane >> 2;
      const bool vlane = vb < sub_boxes;
      const bool boxlane = lane < nbox;
      int id_cur = boxlane ? fetch_id<TILE>(pp, it, br_v, lane, bs_shift) : 0;
      while (it.valid) {
        const UnitInfo ui = it.ui;
        TileIter<TILE> nx = it;
        nx.advance(pp);
        const int id_next = boxlane ? fetch_id<TILE>(pp, nx, br_v, lane, bs_shift) : 0;
        const int my_row = boxlane ? box_row<TILE>(pp, it, br_v, lane, id_cur, bs_shift) : 0;
        const CUtensorMap* map = ui.current ? &tm_cur_v : &tm_kv_v;
        uint8_t* dst = sV8 + vc * L::kV8Chunk + vb * br_v * 128;
        for (int sub = 0; sub < TILE / L::kV8Sub; ++sub) {
          const int st = vs % L::kNV8;
          const int row = __shfl_sync(0xffffffffu, my_row, (sub * sub_boxes + vb) & 7);
          if (vs >= L::kNV8 && !wait(&bar[F_V8EMPTY + st], ((vs / L::kNV8) - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar[F_V8FULL + st], L::kV8Stage);
          if (vlane) tma_load_2d(dst + st * L::kV8Stage, map, &bar[F_V8FULL + st], vc * 128, row);
          ++vs;
        }
        if (!ok) break;
        id_cur = id_next;
        it = nx;
      }
      if (lane == 0)
        for (int s = 0; s < L::kNV8 && s < vs; ++s) {
          const int last = vs - 1 - ((vs - 1 - s) % L::kNV8);
          mbar_wait(&bar[F_V8FULL + s], (last / L::kNV8) & 1, err);
        }
    } else if (warp == 1) {
      // ------------------------------------------------ rank 1: MMA issuer (PV)
      if (lane == 0) {
        // E4M3 x E4M3 -> fp32; P K-major, V MN-major (latent-contiguous rows)
        constexpr uint32_t idesc = make_idesc_f16(128, 256, false, false, true);
        const uint32_t v_base = smem_u32(sV8);
        const uint32_t p_base = smem_u32(sPr);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0, vs = 0, nfix = 0;
        bool ok = true;
        while (ok && it.valid) {
          const int sb = g & 1;
          if (!wait(&bar[F_P8_READY + sb], (g >> 1) & 1)) break;
          const uint32_t hdr =
              *reinterpret_cast<volatile uint32_t*>(sPr + sb * L::kMsgStride + L::kMsgHdr);
          const bool first = it.first();
          if (first && it.k >= 1 && !wait(&bar[F_O_EMPTY], (it.k - 1) & 1)) break;
          if (hdr & 1u) {
            if (!wait(&bar[F_O_FIXED], nfix & 1)) break;
            ++nfix;
          }
          const uint32_t pa = p_base + sb * L::kMsgStride;
          for (int sub = 0; sub < TILE / L::kV8Sub; ++sub) {
            const int st = vs % L::kNV8;
            if (!wait(&bar[F_V8FULL + st], (vs / L::kNV8) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t vb = v_base + st * L::kV8Stage;
#pragma unroll
            for (int kk = 0; kk < L::kV8Sub / 32; ++kk) {
#pragma unroll
              for (int term = 0; term < 2; ++term) {
                // tokens [64 sub + 32 kk, +32) of the hi (bytes 0..63) or lo
                // (bytes 64..127) half of the rows of tile `sub`
                const uint64_t ad = make_desc_sw128(pa + sub * 16384 + term * 64 + kk * 32, 16, 1024);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                  const uint64_t bd = make_desc_sw128(vb + half * 2 * L::kV8Chunk + kk * 32 * 128,
                                                      L::kV8Chunk, 1024);
                  umma_ss_f8(tmem + half * 256, ad, bd, idesc,
                             (first && sub == 0 && kk == 0 && term == 0) ? 0u : 1u);
                }
              }
            }
            umma_commit(&bar[F_V8EMPTY + st]);
            ++vs;
          }
          if (!ok) break;
          umma_commit(&bar[F_PV_DONE + sb]);
          it.advance(pp);
          ++g;
        }
        umma_commit(&bar[F_MMA_DONE_B]);
        mbar_wait(&bar[F_MMA_DONE_B], 0, err);
      }
    } else if (warp == 2) {
      // ------------------------------------------------ rank 1: hand P buffers back
      if (lane == 0) {
        const uint32_t pfree_peer = map_to_peer(&bar[F_PFREE], 0);
        TileIter<TILE> it;
        it.start(pp, rng);
        int g = 0;
        while (it.valid) {
          const int sb = g & 1;
          if (!wait(&bar[F_PV_DONE + sb], (g >> 1) & 1)) break;
          if (!wait(&bar[F_META_READ + sb], (g >> 1) & 1)) break;
          mbar_arrive_expect_tx(&bar[F_P_FULL + sb], L::kMsgBytes);   // tile g + 2
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
    } else {
      // ------------------------------------------------ rank 1: O rescale + epilogue
      // group k: latent columns [k kOCols, (k + 1) kOCols) of row r
      const int grp = (warp - 4) >> 2;
      const int r = (threadIdx.x - 128) & 127;
      const int wq = warp & 3;
      const int cbeg = kOCols * grp;
      const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
      TileIter<TILE> it;
      it.start(pp, rng);
      int g = 0;
      bool ok = true;
      while (ok && it.valid) {
        const UnitInfo ui = it.ui;
        const int sb = g & 1;
        if (!wait_lazy(&bar[F_P_FULL + sb], (g >> 1) & 1)) { ok = false; break; }
        if (threadIdx.x == 128) *msg_count = g + 1;   // messages seen to land (for the drain)
        uint8_t* msg = sPr + sb * L::kMsgStride;
        const uint32_t hdr = *reinterpret_cast<const volatile uint32_t*>(msg + L::kMsgHdr);
        const float alpha = reinterpret_cast<const float*>(msg + L::kMsgAlpha)[r];
        const float lsum = reinterpret_cast<const float*>(msg + L::kMsgLA)[r] +
                           reinterpret_cast<const float*>(msg + L::kMsgLB)[r];
        const float m2 = reinterpret_cast<const float*>(msg + L::kMsgM)[r];
#pragma unroll 1
        for (int tile = grp * (2 / kGroups); tile < (grp + 1) * (2 / kGroups); ++tile) {
          // row r of 64-token tile `tile`: fp16 p' -> [hi bytes | lo bytes]
          // in the same 128-byte row (each thread rewrites only its own row)
          uint8_t* row = msg + tile * 16384;
          uint4 x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] = *reinterpret_cast<const uint4*>(row + sw128_offset(r, u));
          uint32_t hw[16], lw[16];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
            uint32_t h[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_e4m3x2(w[e], h[e], lo[e]);
            hw[2 * u] = h[0] | (h[1] << 16);
            hw[2 * u + 1] = h[2] | (h[3] << 16);
            lw[2 * u] = lo[0] | (lo[1] << 16);
            lw[2 * u + 1] = lo[2] | (lo[3] << 16);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            *reinterpret_cast<uint4*>(row + sw128_offset(r, u)) =
                make_uint4(hw[4 * u], hw[4 * u + 1], hw[4 * u + 2], hw[4 * u + 3]);
            *reinterpret_cast<uint4*>(row + sw128_offset(r, 4 + u)) =
                make_uint4(lw[4 * u], lw[4 * u + 1], lw[4 * u + 2], lw[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[F_P8_READY + sb]);
        // the message's header fields are in registers: the slot may go back
        // (once the PV MMAs have read its P as well)
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[F_META_READ + sb]);
        if (hdr & 1u) {
          // O *= alpha before PV of this tile; PV of the previous tile must be done
          if (!wait_lazy(&bar[F_PV_DONE + ((g - 1) & 1)], ((g - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          rescale_o<kOCols>(tmem + lane_base, cbeg, alpha);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[F_O_FIXED]);
        }
        if (hdr & 2u) {
          // epilogue of the piece: O * kv_scale / (2^6 l) and its LSE
          if (!wait_lazy(&bar[F_PV_DONE + sb], (g >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const float lse2 = m2 + __log2f(lsum) - static_cast<float>(kPShift);   // log2 domain
          const float mul = pp.out_scale / lsum;   // lsum is the row sum of p' = 2^6 p
          const int64_t row_out =
              part_row(pp, static_cast<int64_t>(ui.b) * pp.q_len + ui.i, ui.p, r);   // r < H only
          // whole unit: o_part rows; a piece of a unit split across pairs:
          // O / l and the LSE (log2) parked in this pair's workspace slot for
          // the merge kernel
          const bool whole = it.whole();
          const int slot = 2 * cid + (it.u == rng.u_begin ? 0 : 1);
          if (whole)
            store_o_half<kOCols>(tmem + lane_base, cbeg, pp.o_part, row_out * 512, mul, pp.part_dtype,
                         r < pp.H);
          else
            store_o_half<kOCols>(tmem + lane_base, cbeg, pp.ws_o, (static_cast<int64_t>(slot) * 128 + r) * 512,
                         mul, pp.part_dtype, true);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[F_O_EMPTY]);
          if (grp == 0) {
            if (!whole) pp.ws_lse[slot * 128 + r] = lse2;
            else if (r < pp.H) pp.lse_part[row_out] = lse2 * kLn2;
          }
        }
        it.advance(pp);
        ++g;
      }
    }
  }

  // every tensor-memory access of this thread has completed before TMEM is freed
  __syncwarp();
  tmem_wait_st();
  tmem_wait_ld();
  tc_fence_before();
  __syncthreads();
  if (pp.split && rank == 1 && threadIdx.x == 0) record_split_unit<TILE>(pp, cid, rng, shares, split);
  cluster_sync();
  if (rank == 1 && threadIdx.x == 64) {
    // Drain the P messages rank 0 sent that the epilogue warps never saw
    // land (they stop early when a wait runs out): rank 1 must not exit while
    // rank 0's stores still write here.  Every message went to an armed slot,
    // so each complete one completes a P_FULL phase.
    const uint32_t sent_addr = map_to_peer(const_cast<int*>(msg_count), 0);
    int sent;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sent) : "r"(sent_addr) : "memory");
    for (int k = *msg_count; k < sent; ++k) mbar_wait(&bar[F_P_FULL + (k & 1)], (k >> 1) & 1, err);
  }
  cluster_sync();   // no DSMEM traffic into either CTA after this point
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- launcher
// Shared-memory limit and co-resident pairs of the kernel on the current
// device (cached per device ordinal under a lock, as for the 16-bit kernel).
template <bool BF16>
static int prepare_partial_fp8(int* clusters) {
  static int cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    auto kern = mla_partial_fp8_kernel<BF16>;
    constexpr int smem = Fp8Smem::kTotal;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kFp8Threads, 1, 1);
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
    cache[dev] = std::min(mc, 256);
  }
  *clusters = cache[dev];
  return 0;
}

int partial_fp8_max_clusters() {
  int a = 0, b = 0;
  if (prepare_partial_fp8<true>(&a) != 0 || prepare_partial_fp8<false>(&b) != 0) return -1;
  return std::min(a, b);
}

template <bool BF16>
static int launch_partial_fp8_t(const CUtensorMap& qlat, const CUtensorMap& qpe,
                                const CUtensorMap& kv, const CUtensorMap& cur,
                                const CUtensorMap& kv_v, const CUtensorMap& cur_v,
                                const PartialParams& pp, cudaStream_t stream) {
  int max_clusters = 0;
  if (prepare_partial_fp8<BF16>(&max_clusters) != 0) return -1;
  const int clusters = pp.split ? pp.split : std::max(1, std::min(pp.num_units, max_clusters));
  if (clusters > max_clusters) return -1;
  mla_partial_fp8_kernel<BF16><<<dim3(2 * clusters), dim3(kFp8Threads), Fp8Smem::kTotal, stream>>>(
      qlat, qpe, kv, cur, kv_v, cur_v, pp);
  return pp.split ? launch_partial_merge(pp, clusters, stream) : 0;
}

int launch_partial_fp8(const CUtensorMap& qlat, const CUtensorMap& qpe, const CUtensorMap& kv,
                       const CUtensorMap& cur, const CUtensorMap& kv_v, const CUtensorMap& cur_v,
                       const PartialParams& pp, bool bf16, cudaStream_t stream) {
  return bf16 ? launch_partial_fp8_t<true>(qlat, qpe, kv, cur, kv_v, cur_v, pp, stream)
              : launch_partial_fp8_t<false>(qlat, qpe, kv, cur, kv_v, cur_v, pp, stream);
}

}  // namespace mla
