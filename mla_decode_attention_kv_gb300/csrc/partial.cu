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
// query heads of token i as the M dimension:
//   S = Q . K^T        Q [128 x 576], K = tile of TILE cached tokens x 576
//   P = exp2(S*scale*log2e - m)    (online softmax, running max m, lazy rescale)
//   O += P . V         V = the same tile's latent columns, [TILE x 512]
//
// GB300 mapping.  A 128 x 512 fp32 accumulator alone fills an SM's whole
// tensor memory (128 lanes x 512 columns), so each unit runs on a CLUSTER OF
// TWO CTAs on two SMs:
//   CTA 0 owns latent chunks 0..3 (dims 0..255) and the RoPE chunk (512..575)
//   CTA 1 owns latent chunks 4..7 (dims 256..511)
// Each CTA TMA-loads only its own 64-dim chunks of Q and of every KV tile, so
// each KV byte crosses HBM exactly once.  Each CTA computes the partial
// S_r = Q_r . K_r^T over its chunks on its tensor cores; the two fp32
// partials are swapped through distributed shared memory and summed, so both
// CTAs hold the same S, take the same softmax and produce the same P.  Each
// CTA then accumulates its 256-column half of O = P . V_r in TMEM.
//
// Roles per CTA (256 threads):
//   warp 0       TMA producer: Q once per unit, KV tiles into a STAGES ring
//   warp 1       MMA issuer (tcgen05, one elected thread); owns TMEM
//   warps 4..7   softmax + S exchange + O rescale + epilogue (thread = head)
// Every wait is bounded; on timeout the kernel records MLA_DEV_WAIT_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

// Token range of one unit.  History shard p of sequence b covers
// [p*len, min(L, (p+1)*len)), len = bs * ceil(L / (S*bs)) (block-aligned,
// trailing shards possibly empty).  The CURRENT part covers kv_cur[b, 0..i].
struct UnitInfo {
  int b, i, p;
  int lo, hi;      // token range inside the part's token space
  bool current;
  int ntiles;
};

template <int TILE>
__device__ __forceinline__ UnitInfo unit_info(const PartialParams& pp, int u) {
  UnitInfo ui;
  ui.i = u % pp.q_len;
  int bp = u / pp.q_len;
  ui.p = bp % pp.P;
  ui.b = bp / pp.P;
  ui.current = pp.has_cur && ui.p == pp.S;
  if (ui.current) {
    ui.lo = 0;
    ui.hi = ui.i + 1;
  } else {
    int L = pp.seq_lens[ui.b];
    L = max(0, min(L, pp.max_blocks * pp.bs));
    int chunk = pp.S * pp.bs;
    int len = L > 0 ? pp.bs * ((L + chunk - 1) / chunk) : 0;
    ui.lo = min(L, ui.p * len);
    ui.hi = min(L, (ui.p + 1) * len);
  }
  ui.ntiles = (ui.hi - ui.lo + TILE - 1) / TILE;
  return ui;
}

template <int TILE, int STAGES>
struct PartialSmem {
  static constexpr int kChunks = 5;                       // CTA 0: 4 latent + RoPE
  static constexpr int kQBytes = kChunks * 128 * 128;     // 80 KB
  static constexpr int kChunkBytes = TILE * 128;          // one 64-dim chunk of a tile
  static constexpr int kStageBytes = kChunks * kChunkBytes;
  static constexpr int kPBytes = TILE == 32 ? 16384 : 32768;   // two P buffers
  static constexpr int kXBytes = 128 * TILE * 4;          // one exchange buffer
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBytes;
  static constexpr int kPOff = kKVOff + STAGES * kStageBytes;
  static constexpr int kXOff = kPOff + kPBytes;
  static constexpr int kBarOff = kXOff + 2 * kXBytes;
  static constexpr int kTotal = kBarOff + 256 + 1024;     // barriers + 1 KB align slack
};

template <int TILE, int STAGES, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tm_qabs,
                       const __grid_constant__ CUtensorMap tm_qpe,
                       const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_cur, const PartialParams pp) {
  using L = PartialSmem<TILE, STAGES>;
  static_assert(TILE == 32 || TILE == 64, "TILE");
  static_assert(L::kTotal <= 232448, "shared memory budget");
  constexpr int kTmemCols = 512;
  constexpr uint32_t kOCol = 0;          // O half: columns [0, 256)
  constexpr uint32_t kSCol = 256;        // S buffers: [256, 256 + 2*TILE)
  constexpr float kRescaleThresh = 8.0f; // lazy rescale: only when max grows by > 2^8

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sKV = smem + L::kKVOff;
  uint8_t* sP = smem + L::kPOff;
  uint8_t* sX = smem + L::kXOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* kv_full = bars;                 // [STAGES]
  uint64_t* kv_empty = bars + STAGES;       // [STAGES]
  uint64_t* q_full = bars + 2 * STAGES;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;            // [2]
  uint64_t* s_empty = q_full + 4;           // [2]
  uint64_t* p_full = q_full + 6;            // [2]
  uint64_t* p_empty = q_full + 8;           // [2]
  uint64_t* x_full = q_full + 10;           // [2]  arrived by the peer
  uint64_t* x_empty = q_full + 12;          // [2]  arrived by the peer
  uint64_t* o_empty = q_full + 14;
  uint64_t* mma_done = q_full + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(q_full + 17);

  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;        // chunks owned by this CTA
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = pp.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&s_empty[k], 4);
      mbar_init(&p_full[k], 4);
      mbar_init(&p_empty[k], 1);
      mbar_init(&x_full[k], 4);
      mbar_init(&x_empty[k], 4);
    }
    mbar_init(o_empty, 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_qabs);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_kv);
    prefetch_tmap(&tm_cur);
  }
  __syncthreads();
  cluster_sync();  // peer barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(nclusters_x());

  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((it & 1023u) == 1023u && *abort_flag) return false;
    }
    set_error(err, kDevWaitTimeout);
    *abort_flag = 1;
    return false;
  };
  auto wait_cl = [&](uint64_t* bar, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      if (mbar_try_wait_cluster(bar, parity)) return true;
      if ((it & 1023u) == 1023u && *abort_flag) return false;
    }
    set_error(err, kDevWaitTimeout);
    *abort_flag = 1;
    return false;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();   // KV is read once
      const uint64_t pol_keep = policy_evict_last();      // Q is shared by units
      int g = 0, k = 0;
      int last_g[STAGES];
      for (int s = 0; s < STAGES; ++s) last_g[s] = -1;
      int q_issued = 0;
      bool ok = true;
      for (int u = cid; u < pp.num_units && ok; u += ncl) {
        UnitInfo ui = unit_info<TILE>(pp, u);
        if (ui.ntiles == 0) continue;
        if (k >= 1 && !wait(q_empty, (k - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, nch * 16384);
        const int qrow = (ui.b * pp.q_len + ui.i) * pp.H;
        for (int c = 0; c < nch; ++c) {
          if (rank == 0 && c == 4)
            tma_load_2d(sQ + c * 16384, &tm_qpe, q_full, 0, qrow, pol_keep);
          else
            tma_load_2d(sQ + c * 16384, &tm_qabs, q_full, (rank * 4 + c) * 64, qrow, pol_keep);
        }
        q_issued = k + 1;
        for (int j = 0; j < ui.ntiles; ++j, ++g) {
          const int st = g % STAGES;
          if (g >= STAGES && !wait(&kv_empty[st], ((g / STAGES) - 1) & 1)) { ok = false; break; }
          uint8_t* dst = sKV + st * L::kStageBytes;
          mbar_arrive_expect_tx(&kv_full[st], nch * L::kChunkBytes);
          const int t0 = ui.lo + j * TILE;
          for (int sub = 0; sub < TILE / pp.box_rows; ++sub) {
            int row;
            const CUtensorMap* map;
            if (ui.current) {
              row = ui.b * pp.q_len + sub * pp.box_rows;
              map = &tm_cur;
            } else {
              int t = t0 + sub * pp.box_rows;
              // sub-boxes past the unit's last token re-read its last page
              // (in bounds, finite, masked out by the softmax)
              if (t >= ui.hi) t = ui.hi - 1;
              const int lb = t / pp.bs;
              int pb = pp.block_table[static_cast<int64_t>(ui.b) * pp.max_blocks + lb];
              if (pb < 0 || pb >= pp.num_blocks) {
                set_error(err, kDevBadBlockId);
                pb = 0;
              }
              row = pb * pp.bs + (t % pp.bs);
              if (t != t0 + sub * pp.box_rows) row -= row % pp.box_rows;
              map = &tm_kv;
            }
            for (int c = 0; c < nch; ++c) {
              const int x = (rank == 0 && c == 4) ? 512 : (rank * 4 + c) * 64;
              tma_load_2d(dst + c * L::kChunkBytes + sub * pp.box_rows * 128, map, &kv_full[st], x,
                          row, pol_stream);
            }
          }
          last_g[st] = g;
        }
        ++k;
      }
      // drain: every issued copy has landed before this CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (last_g[s] >= 0) mbar_wait(&kv_full[s], (last_g[s] / STAGES) & 1, err);
      if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16(128, TILE, BF16, false, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(128, 256, BF16, false, true);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      const uint32_t p_base = smem_u32(sP);
      int g = 0, k = 0;
      bool ok = true;
      auto issue_pv = [&](int gg, bool first) -> bool {
        const int sb = gg & 1;
        if (!wait(&p_full[sb], (gg >> 1) & 1)) return false;
        if (first && k >= 1 && !wait(o_empty, (k - 1) & 1)) return false;
        tc_fence_after();
        const int st = gg % STAGES;
        const uint32_t v_base = kv_base + st * L::kStageBytes;
        const uint32_t pa = p_base + (TILE == 32 ? sb * 64 : sb * 16384);
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk) {
          const uint64_t ad = make_desc_sw128(pa + kk * 32, 16, 1024);
          const uint64_t bd = make_desc_sw128(v_base + kk * 2048, L::kChunkBytes, 1024);
          umma_ss(tmem + kOCol, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(&p_empty[sb]);
        umma_commit(&kv_empty[st]);
        return true;
      };
      for (int u = cid; u < pp.num_units && ok; u += ncl) {
        UnitInfo ui = unit_info<TILE>(pp, u);
        if (ui.ntiles == 0) continue;
        if (!wait(q_full, k & 1)) { ok = false; break; }
        const int g0 = g;
        for (int j = 0; j < ui.ntiles; ++j, ++g) {
          const int st = g % STAGES;
          const int sb = g & 1;
          if (!wait(&kv_full[st], (g / STAGES) & 1)) { ok = false; break; }
          if (g >= 2 && !wait(&s_empty[sb], ((g >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kv_st = kv_base + st * L::kStageBytes;
          for (int c = 0; c < nch; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_desc_sw128(q_base + c * 16384 + kk * 32, 16, 1024);
              const uint64_t bd = make_desc_sw128(kv_st + c * L::kChunkBytes + kk * 32, 16, 1024);
              umma_ss(tmem + kSCol + sb * TILE, ad, bd, idesc_qk, (c | kk) ? 1u : 0u);
            }
          }
          umma_commit(&s_full[sb]);
          if (j == ui.ntiles - 1) umma_commit(q_empty);
          if (j >= 1 && !issue_pv(g - 1, j - 1 == 0)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(g - 1, ui.ntiles == 1)) { ok = false; break; }
        (void)g0;
        ++k;
      }
      // drain: all MMAs of this thread complete before TMEM is released
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, err);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x - 128;             // TMEM lane == query head
    const int wq = warp & 3;                     // TMEM lane quarter of this warp
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t x_peer = map_to_peer(sX, peer);
    const uint32_t xfull_peer0 = map_to_peer(&x_full[0], peer);
    const uint32_t xempty_peer0 = map_to_peer(&x_empty[0], peer);
    uint8_t* my_x = sX;
    int g = 0, k = 0;
    bool ok = true;
    for (int u = cid; u < pp.num_units && ok; u += ncl) {
      UnitInfo ui = unit_info<TILE>(pp, u);
      const int64_t row_out =
          (static_cast<int64_t>(ui.b * pp.q_len + ui.i) * pp.P + ui.p) * pp.H + r;
      if (ui.ntiles == 0) {
        // empty part: o = 0, lse = -inf
        if (r < pp.H) {
          for (int c = 0; c < 256; c += 8) {
            const int64_t e = row_out * 512 + rank * 256 + c;
            if (pp.part_dtype == 2) {
              float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
              reinterpret_cast<float4*>(static_cast<float*>(pp.o_part) + e)[0] = z;
              reinterpret_cast<float4*>(static_cast<float*>(pp.o_part) + e)[1] = z;
            } else {
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(pp.o_part) + e) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          if (rank == 0) pp.lse_part[row_out] = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY;   // running max, log2 domain
      float l = 0.f;         // running sum of exp2(x - m)
      for (int j = 0; j < ui.ntiles; ++j, ++g) {
        const int sb = g & 1;
        const int nvalid = min(TILE, ui.hi - (ui.lo + j * TILE));
        if (!wait(&s_full[sb], (g >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float s[TILE];
#pragma unroll
        for (int c0 = 0; c0 < TILE; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kSCol + sb * TILE + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) s[c0 + t] = __uint_as_float(v[t]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sb]);

        // ---- swap partial S with the peer CTA (fp32, swizzled rows)
        if (g >= 2 && !wait_cl(&x_empty[sb], ((g >> 1) - 1) & 1)) { ok = false; break; }
        const uint32_t xrow_peer = x_peer + sb * L::kXBytes + r * (TILE * 4);
#pragma unroll
        for (int uu = 0; uu < TILE / 4; ++uu)
          st_cluster_v4(xrow_peer + ((uu ^ (r & 7)) << 4), s[4 * uu], s[4 * uu + 1],
                        s[4 * uu + 2], s[4 * uu + 3]);
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          mbar_arrive_remote(xfull_peer0 + sb * 8);
        }
        if (!wait_cl(&x_full[sb], (g >> 1) & 1)) { ok = false; break; }
        const uint8_t* xrow = my_x + sb * L::kXBytes + r * (TILE * 4);
#pragma unroll
        for (int uu = 0; uu < TILE / 4; ++uu) {
          const float4 o4 = *reinterpret_cast<const float4*>(xrow + ((uu ^ (r & 7)) << 4));
          s[4 * uu] += o4.x;
          s[4 * uu + 1] += o4.y;
          s[4 * uu + 2] += o4.z;
          s[4 * uu + 3] += o4.w;
        }
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          mbar_arrive_remote(xempty_peer0 + sb * 8);
        }

        // ---- online softmax (log2 domain)
        float mt = -INFINITY;
#pragma unroll
        for (int t = 0; t < TILE; ++t) {
          bool valid = t < nvalid;
          if (ui.current) valid = t <= ui.i;
          s[t] = valid ? s[t] * pp.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[t]);
        }
        bool need_rescale = false;
        float alpha = 1.f;
        if (j == 0) {
          m = mt;
        } else if (mt > m + kRescaleThresh) {
          need_rescale = true;
          alpha = fast_exp2(m - mt);
          m = mt;
        }
        float psum = 0.f;
#pragma unroll
        for (int t = 0; t < TILE; ++t) {
          s[t] = fast_exp2(s[t] - m);   // masked: exp2(-inf) = 0
          psum += s[t];
        }
        l = l * alpha + psum;

        // O rescale (rare): needs PV of the previous tile complete
        if (__any_sync(0xffffffffu, need_rescale)) {
          if (!wait(&p_empty[(g - 1) & 1], ((g - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          for (int c0 = 0; c0 < 256; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kOCol + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
            tmem_st32(tmem + lane_base + kOCol + c0, v);
          }
          tmem_wait_st();
        }

        // ---- P (bf16 / fp16, swizzled K-major rows) for the PV MMA
        if (g >= 2 && !wait(&p_empty[sb], ((g >> 1) - 1) & 1)) { ok = false; break; }
        uint8_t* prow = sP + (TILE == 32 ? 0 : sb * 16384);
        const int ubase = TILE == 32 ? sb * 4 : 0;
#pragma unroll
        for (int uu = 0; uu < TILE / 8; ++uu) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) w[e] = pack2<BF16>(s[8 * uu + 2 * e], s[8 * uu + 2 * e + 1]);
          *reinterpret_cast<uint4*>(prow + sw128_offset(r, ubase + uu)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!ok) break;

      // ---- epilogue: O / l -> o_part, lse -> lse_part
      const int gl = g - 1;
      if (!wait(&p_empty[gl & 1], (gl >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.f / l;
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kOCol + c0, v);
        tmem_wait_ld();
        if (r < pp.H) {
          const int64_t e = row_out * 512 + rank * 256 + c0;
          store_row32(pp.o_part, e, v, inv_l, pp.part_dtype);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      if (rank == 0 && r < pp.H) pp.lse_part[row_out] = (m + __log2f(l)) * 0.6931471805599453f;
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no remote access into this CTA's smem after this point
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- launcher
template <int TILE, int STAGES, bool BF16>
static int launch_partial_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                            const CUtensorMap& d, const PartialParams& pp, cudaStream_t stream) {
  auto kern = mla_partial_kernel<TILE, STAGES, BF16>;
  constexpr int smem = PartialSmem<TILE, STAGES>::kTotal;
  static bool configured = false;
  static int max_clusters = 0;
  if (!configured) {
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
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess ||
        max_clusters < 1) {
      cudaGetLastError();
      max_clusters = 64;
    }
    configured = true;
  }
  const int clusters = std::max(1, std::min(pp.num_units, max_clusters));
  kern<<<dim3(2 * clusters), dim3(256), smem, stream>>>(a, b, c, d, pp);
  return 0;
}

int launch_partial(const CUtensorMap& qabs, const CUtensorMap& qpe, const CUtensorMap& kv,
                   const CUtensorMap& cur, const PartialParams& pp, bool bf16,
                   cudaStream_t stream) {
  return bf16 ? launch_partial_t<kPartialTile, 4, true>(qabs, qpe, kv, cur, pp, stream)
              : launch_partial_t<kPartialTile, 4, false>(qabs, qpe, kv, cur, pp, stream);
}

}  // namespace mla
