// LSE combine (mla_lse_combine) and batch-major V-up (mla_vup,
// mla_lse_combine_vup).
//
// Combine (vllm-ascend PR #16977 study page: glossary "LSE"; the fourth
// change, where all history shards and the local CURRENT partial are merged
// exactly once and the local partial is read in place): for row (t, h)
//   LSE = ln sum_p exp(lse_p),   o = sum_p exp(lse_p - LSE) * o_p.
// Partials are read in their own dtype (bf16 / fp16 / fp32) with no fp32
// copy (same page, first change: dtype pass-through); parts with lse = -inf
// are skipped; parts are visited in index order, then the local one.
//
// V-up (same page, code block A, _v_up_proj_batch_major): the latent output
// stays batch-major [T, H, 512]; each head is multiplied by W_UV[h]
// (512 x 128) and the result is stored as [T, H*128].  Here it is one
// tcgen05 GEMM per head on GB300 tensor cores:
//   D[v, t] = sum_k W_UV[h][k, v] * o[t, h, k]
// A = W_UV[h]^T (M = 128 v-columns, MN-major straight from W_UV's rows,
// TMA-loaded), B = the latent rows of head h (N = rows of a 64-row tile,
// K-major in shared memory), D in TMEM.  In the fused form the combine writes
// its bf16/fp16 result for head h directly into that B operand.
//
// When the partials are stored in W_UV's dtype the fused call instead takes
// the up-projection of every part and the LSE-weighted sum afterwards, in the
// 128-wide V space (the projection is linear):
//   out[t, h] = sum_p w_p(t, h) * (o_p[t, h, :] . W_UV[h]),  w_p = exp(lse_p - LSE)
// so the partials go from global memory to the tensor cores by TMA with no
// pass through registers (mla_vup_parts_kernel).
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

// ---------------------------------------------------------------- weights
// Normalised weights of the parts of row (t, h), spread over the warp: lane
// l holds the weights of parts l, l + 32 and l + 64 (zero for empty parts).
// Part index P (when a local partial is given) is the local one.
struct RowWeights {
  float w[3];
  float lse;
};

__device__ __forceinline__ RowWeights row_weights(const float* lse_part, int P, int H, int64_t t,
                                                  int h, const float* lse_local, int lane) {
  const int np = P + (lse_local ? 1 : 0);
  RowWeights rw;
  float v[3];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int p = lane + 32 * k;
    v[k] = -INFINITY;
    if (p < np) v[k] = p < P ? __ldg(lse_part + (t * P + p) * H + h) : __ldg(lse_local + t * H + h);
    mx = fmaxf(mx, v[k]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    v[k] = (mx == -INFINITY || v[k] == -INFINITY) ? 0.f : __expf(v[k] - mx);
    sum += v[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) rw.w[k] = v[k] * inv;
  rw.lse = sum > 0.f ? mx + __logf(sum) : -INFINITY;
  return rw;
}

__device__ __forceinline__ float weight_of(const RowWeights& rw, int p) {
  const float x = p < 32 ? rw.w[0] : (p < 64 ? rw.w[1] : rw.w[2]);
  return __shfl_sync(0xffffffffu, x, p & 31);
}

// 16 consecutive elements of one partial row: 64 bytes (fp32) or 32 bytes.
template <bool F32>
struct Chunk16 {
  uint4 v[F32 ? 4 : 2];
};

template <bool F32>
__device__ __forceinline__ Chunk16<F32> load16(const void* src, int64_t e) {
  Chunk16<F32> x;
  const uint4* p = F32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(src) + e)
                       : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + e);
#pragma unroll
  for (int i = 0; i < (F32 ? 4 : 2); ++i) x.v[i] = __ldg(p + i);
  return x;
}

template <bool F32>
__device__ __forceinline__ void fma16(const Chunk16<F32>& x, int dt, float w, float (&acc)[16]) {
  if constexpr (F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[4 * i] += w * __uint_as_float(x.v[i].x);
      acc[4 * i + 1] += w * __uint_as_float(x.v[i].y);
      acc[4 * i + 2] += w * __uint_as_float(x.v[i].z);
      acc[4 * i + 3] += w * __uint_as_float(x.v[i].w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t u[4] = {x.v[i].x, x.v[i].y, x.v[i].z, x.v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = unpack2(u[k], dt);
        acc[8 * i + 2 * k] += w * f.x;
        acc[8 * i + 2 * k + 1] += w * f.y;
      }
    }
  }
}

// Combine NR rows (t[0..NR)) of head h for this lane's 16 latent elements.
// All loads of a batch of parts are issued before any of them is used.
template <int NR, bool F32>
__device__ __forceinline__ void combine_rows(const void* o_part, const float* lse_part, int P,
                                             const void* o_local, const float* lse_local, int H,
                                             const int64_t (&t)[NR], const bool (&valid)[NR],
                                             int h, int dt, int lane, float (&acc)[NR][16],
                                             float (&lse)[NR]) {
  constexpr int KB = F32 ? 4 : 8;   // parts per batch
  RowWeights rw[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    rw[r] = row_weights(lse_part, P, H, valid[r] ? t[r] : 0, h, lse_local, lane);
    lse[r] = rw[r].lse;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[r][i] = 0.f;
  }
  const int np = P + (o_local ? 1 : 0);
  for (int p0 = 0; p0 < np; p0 += KB) {
    Chunk16<F32> x[NR][KB];
    float w[NR][KB];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const int p = p0 + k;
        w[r][k] = p < np ? weight_of(rw[r], p) : 0.f;
        if (valid[r] && w[r][k] != 0.f) {
          const void* src = p < P ? o_part : o_local;
          const int64_t row = p < P ? (t[r] * P + p) * H + h : t[r] * H + h;
          x[r][k] = load16<F32>(src, row * 512 + lane * 16);
        } else {
#pragma unroll
          for (int i = 0; i < (F32 ? 4 : 2); ++i) x[r][k].v[i] = make_uint4(0, 0, 0, 0);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
#pragma unroll
      for (int k = 0; k < KB; ++k)
        if (w[r][k] != 0.f) fma16<F32>(x[r][k], dt, w[r][k], acc[r]);
    }
  }
}

__device__ __forceinline__ void store16(void* dst, int64_t e, const float (&v)[16], int dt) {
  if (dt == kFP32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(dst) + e);
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + e);
#pragma unroll
    for (int q = 0; q < 2; ++q)
      p[q] = make_uint4(pack2_dt(v[8 * q], v[8 * q + 1], dt), pack2_dt(v[8 * q + 2], v[8 * q + 3], dt),
                        pack2_dt(v[8 * q + 4], v[8 * q + 5], dt),
                        pack2_dt(v[8 * q + 6], v[8 * q + 7], dt));
  }
}

// ---------------------------------------------------------------- combine
// One warp per (t, h) row; lane l owns latent elements [16l, 16l + 16).
template <bool F32>
__global__ void __launch_bounds__(256) mla_combine_kernel(const void* o_part, const float* lse_part,
                                                          int P, const void* o_local,
                                                          const float* lse_local, int T, int H,
                                                          int part_dt, int out_dt, void* o_latent,
                                                          float* lse_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(T) * H) return;
  const int64_t t[1] = {row / H};
  const bool valid[1] = {true};
  const int h = static_cast<int>(row % H);
  float acc[1][16];
  float lse[1];
  combine_rows<1, F32>(o_part, lse_part, P, o_local, lse_local, H, t, valid, h, part_dt, lane, acc,
                       lse);
  store16(o_latent, row * 512 + lane * 16, acc[0], out_dt);
  if (lse_out && lane == 0) lse_out[row] = lse[0];
}

// ---------------------------------------------------------------- combine of exchanged partials
// Decode context parallelism across GPUs (vllm-ascend PR #16977 study page,
// the third change: the all-to-all of history partials with heads scattered,
// then the combine of all shards plus the local partial exactly once).  After
// a head-scattered all-to-all every rank holds, for its slice of H heads,
// the partials of all nsrc ranks as [nsrc][T][P][H] rows.  Parts
// (src, p < hist) are every rank's history shards; the CURRENT partial
// (part hist, computed by every rank alike) is taken once, from source
// local_src.  One warp per (t, h) row, lane l owns elements [16l, 16l + 16).
template <bool F32>
__global__ void __launch_bounds__(256) mla_combine_exchanged_kernel(
    const void* o_recv, const float* lse_recv, int nsrc, int P, int hist, int local_src, int T,
    int H, int part_dt, int out_dt, void* o_latent, float* lse_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(T) * H) return;
  const int64_t t = row / H;
  const int h = static_cast<int>(row % H);
  const int nh = nsrc * hist;
  const int np = nh + (local_src >= 0 ? 1 : 0);
  auto part_row = [&](int q) -> int64_t {
    const int src = q < nh ? q / hist : local_src;
    const int p = q < nh ? q - src * hist : hist;
    return ((static_cast<int64_t>(src) * T + t) * P + p) * H + h;
  };
  // weights: lane l holds parts l, l + 32, l + 64 (np <= 96, checked by the host)
  float v[3];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int q = lane + 32 * k;
    v[k] = q < np ? __ldg(lse_recv + part_row(q)) : -INFINITY;
    mx = fmaxf(mx, v[k]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    v[k] = (mx == -INFINITY || v[k] == -INFINITY) ? 0.f : __expf(v[k] - mx);
    sum += v[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  RowWeights rw;
#pragma unroll
  for (int k = 0; k < 3; ++k) rw.w[k] = v[k] * inv;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  constexpr int KB = F32 ? 4 : 8;   // parts per batch of loads
  for (int q0 = 0; q0 < np; q0 += KB) {
    Chunk16<F32> x[KB];
    float w[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      const int q = q0 + k;
      w[k] = q < np ? weight_of(rw, q) : 0.f;
      if (w[k] != 0.f) {
        x[k] = load16<F32>(o_recv, part_row(q) * 512 + lane * 16);
      } else {
#pragma unroll
        for (int i = 0; i < (F32 ? 4 : 2); ++i) x[k].v[i] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < KB; ++k)
      if (w[k] != 0.f) fma16<F32>(x[k], part_dt, w[k], acc);
  }
  store16(o_latent, row * 512 + lane * 16, acc, out_dt);
  if (lse_out && lane == 0) lse_out[row] = sum > 0.f ? mx + __logf(sum) : -INFINITY;
}

// ---------------------------------------------------------------- V-up
constexpr int kVupRows = 64;                    // rows (N) per MMA tile
constexpr int kVupWBytes = 512 * 128 * 2;       // W_UV[h]: 128 KB
constexpr int kVupBBytes = 8 * kVupRows * 128;  // 8 chunks of 64 rows x 128 B: 64 KB
constexpr int kVupSmem = kVupWBytes + kVupBBytes + 1024;

// One CTA per head.  COMBINE: B rows come from the LSE combine of the
// partials; otherwise they are read from o_latent.
template <bool COMBINE, bool BF16, bool F32>
__global__ void __launch_bounds__(256, 1)
    mla_vup_kernel(const __grid_constant__ CUtensorMap tm_w, const void* o_part,
                   const float* lse_part, int P, const void* o_local, const float* lse_local,
                   const void* o_latent_in, int T, int H, int part_dt, void* out,
                   void* o_latent_out, float* lse_out, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem;
  uint8_t* sB = smem + kVupWBytes;
  __shared__ __align__(8) uint64_t bar_w, bar_mma;
  __shared__ uint32_t tmem_slot;
  const int h = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int dt = BF16 ? kBF16 : kFP16;

  if (threadIdx.x == 0) {
    mbar_init(&bar_w, 1);
    mbar_init(&bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kVupRows);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    // W_UV[h] rows k in [0, 512), columns v in [0, 128): two 64-column groups,
    // each stored as 512 rows of 128 B (MN-major A operand, LBO = 64 KB).
    mbar_arrive_expect_tx(&bar_w, kVupWBytes);
    const uint64_t pol = policy_evict_first();
    for (int g = 0; g < 2; ++g)
      for (int kh = 0; kh < 2; ++kh)
        tma_load_2d(sW + g * 65536 + kh * 32768, &tm_w, &bar_w, g * 64, h * 512 + kh * 256, pol);
  }
  // W_UV does not depend on the previous kernel; the partials do (programmatic
  // dependent launch: wait here for the grid that wrote them)
  griddep_wait();
  constexpr uint32_t idesc = make_idesc_f16(128, kVupRows, BF16, true, false);
  bool ok = true;
  int phase = 0;
  for (int t0 = 0; t0 < T && ok; t0 += kVupRows, phase ^= 1) {
    const int nrows = min(kVupRows, T - t0);
    // ---- B operand: rows t0 .. t0 + 63 of head h, latent K-major, SW128
    const int c = lane >> 2;          // 64-element chunk of this lane's 16 values
    const int u = 2 * (lane & 3);     // first 16-byte unit inside the 128-byte row
    if constexpr (COMBINE) {
      // rows past nrows are left unwritten: their D columns are never stored
      for (int rr = warp * 2; rr < nrows; rr += 16) {
        const int64_t t[2] = {t0 + rr, t0 + rr + 1};
        const bool valid[2] = {rr < nrows, rr + 1 < nrows};
        float acc[2][16];
        float lse[2];
        combine_rows<2, F32>(o_part, lse_part, P, o_local, lse_local, H, t, valid, h, part_dt,
                             lane, acc, lse);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (!valid[q]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[q][i] = 0.f;
          } else {
            if (o_latent_out) store16(o_latent_out, (t[q] * H + h) * 512 + lane * 16, acc[q], dt);
            if (lse_out && lane == 0) lse_out[t[q] * H + h] = lse[q];
          }
          uint32_t wv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) wv[k] = pack2<BF16>(acc[q][2 * k], acc[q][2 * k + 1]);
          *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr + q, u)) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr + q, u + 1)) =
              make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
      }
    } else {
      for (int rr = warp; rr < nrows; rr += 8) {
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const uint16_t*>(o_latent_in) +
              ((t0 + rr) * static_cast<int64_t>(H) + h) * 512 + lane * 16);
          a = __ldg(src);
          b = __ldg(src + 1);
        }
        *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u)) = a;
        *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u + 1)) = b;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 32) {
      if (t0 == 0 && !mbar_wait(&bar_w, 0, err)) ok = false;
      tc_fence_after();
      if (ok) {
        const uint32_t wa = smem_u32(sW), bb = smem_u32(sB);
#pragma unroll 4
        for (int kk = 0; kk < 32; ++kk) {
          const uint64_t ad = make_desc_sw128(wa + kk * 2048, 65536, 1024);
          const uint64_t bd = make_desc_sw128(bb + (kk >> 2) * (kVupRows * 128) + (kk & 3) * 32, 16, 1024);
          umma_ss(tmem, ad, bd, idesc, kk ? 1u : 0u);
        }
      }
      umma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, phase, err)) ok = false;
    tc_fence_after();
    // ---- epilogue: lane v of TMEM = output column h*128 + v; column = row
    {
      const int wq = warp & 3;
      const int v = wq * 32 + lane;
      const int c0 = (warp >> 2) * 32;   // warps 0-3: rows 0-31, warps 4-7: rows 32-63
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(wq * 32) << 16) + c0, r);
      tmem_wait_ld(r);
      uint16_t* o = static_cast<uint16_t*>(out);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int rr = c0 + j;
        if (rr < nrows) {
          const float f = __uint_as_float(r[j]);
          uint16_t bits;
          if constexpr (BF16) {
            __nv_bfloat16 b = __float2bfloat16_rn(f);
            bits = *reinterpret_cast<uint16_t*>(&b);
          } else {
            __half b = __float2half_rn(f);
            bits = *reinterpret_cast<uint16_t*>(&b);
          }
          o[(static_cast<int64_t>(t0 + rr) * H + h) * 128 + v] = bits;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (threadIdx.x == 0) mbar_wait(&bar_w, 0, err);   // never exit with the W copy in flight
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kVupRows);
  }
}

// ---------------------------------------------------------------- V-up of the parts
// One CTA per head.  For each block of TB rows and each 64-wide K chunk the
// producer stages W_UV[h]'s 64 rows (A, MN-major: two 64-column groups) and
// the chunk of every part's TB rows (B, K-major: part p at B rows
// [p*TB, p*TB + TB), rows past T zero-filled), and one elected thread issues
//   D[v, p*TB + t] += sum_k W_UV[h][k, v] * o_p[t0 + t, h, k]
// (M = 128, N = parts * TB in pieces of at most 256).  Warps 2-3 turn the
// block's LSEs into weights; warps 4-7 (thread = v) read D and store
//   out[t0 + t, h*128 + v] = sum_p w_p(t) * D[v, p*TB + t].
struct VupPartsArgs {
  int T, H, P, has_local;
  const float* lse_part;
  const float* lse_local;
  void* out;
  float* lse_out;
  int* err;
  int ns, stage_bytes, bn;
};

template <bool BF16, int TB>
__global__ void __launch_bounds__(256, 1)
    mla_vup_parts_kernel(const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_p,
                         const __grid_constant__ CUtensorMap tm_l, const VupPartsArgs va) {
  constexpr int kChunks = 512 / 64;
  constexpr int kWChunk = 16384;               // 64 k-rows x 128 v, two 8 KB column groups
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_full[4], bar_empty[4], bar_d_full, bar_d_empty,
      bar_wt_full[2], bar_wt_empty[2], bar_mma_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  __shared__ float s_lse[512];     // LSE of part p, row t of the block: [p * TB + t]
  __shared__ float s_w[2][512];    // weights of the block, double-buffered
  const int h = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int np = va.P + va.has_local;
  const int nblk = (va.T + TB - 1) / TB;
  const int total = nblk * kChunks;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < va.ns; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_d_full, 1);
    mbar_init(&bar_d_empty, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_wt_full[b], 1);
      mbar_init(&bar_wt_empty[b], 4);
    }
    mbar_init(&bar_mma_done, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  int ncols = 32;
  while (ncols < va.bn) ncols <<= 1;
  if (warp == 1) {
    tmem_alloc(&tmem_slot, ncols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_p);
    prefetch_tmap(&tm_l);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  auto wait = [&](uint64_t* b, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      if (mbar_try_wait(b, parity)) return true;
      if ((it & 1023u) == 1023u && *abort_flag) return false;
    }
    set_error(va.err, kDevWaitTimeout);
    *abort_flag = 1;
    return false;
  };
  auto wait_lazy = [&](uint64_t* b, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      if (mbar_try_wait_sleep(b, parity, kLazyWaitNs)) return true;
      if ((it & 15u) == 15u && *abort_flag) return false;
    }
    set_error(va.err, kDevWaitTimeout);
    *abort_flag = 1;
    return false;
  };
  const uint32_t stage_tx = kWChunk + static_cast<uint32_t>(np * TB * 128);

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (converged warp)
    const uint64_t pol_w = nblk > 1 ? policy_evict_last() : policy_evict_first();
    const uint64_t pol_p = policy_evict_first();
    auto issue_w = [&](int q) {
      const int s = q % va.ns;
      uint8_t* st = smem + s * va.stage_bytes;
      const int k0 = h * 512 + (q % kChunks) * 64;
      mbar_arrive_expect_tx(&bar_full[s], stage_tx);
      tma_load_2d(st, &tm_w, &bar_full[s], 0, k0, pol_w);
      tma_load_2d(st + kWChunk / 2, &tm_w, &bar_full[s], 64, k0, pol_w);
    };
    // W_UV does not depend on the previous grid: the first stages' W before
    // the wait for the grid that wrote the partials
    const int pre = min(va.ns, total);
    if (lane == 0)
      for (int q = 0; q < pre; ++q) issue_w(q);
    __syncwarp();
    griddep_wait();
    int q = 0;
    for (; q < total; ++q) {
      const int s = q % va.ns;
      if (q >= va.ns) {
        if (!wait(&bar_empty[s], ((q / va.ns) - 1) & 1)) break;
        if (lane == 0) issue_w(q);
        __syncwarp();
      }
      uint8_t* st = smem + s * va.stage_bytes + kWChunk;
      const int c = q % kChunks, t0 = (q / kChunks) * TB;
      for (int p = lane; p < np; p += 32) {
        if (p < va.P)
          tma_load_3d(st + p * TB * 128, &tm_p, &bar_full[s], c * 64, p * va.H + h, t0, pol_p);
        else
          tma_load_3d(st + p * TB * 128, &tm_l, &bar_full[s], c * 64, h, t0, pol_p);
      }
    }
    // drain: W is in flight for every stage armed so far
    const int armed = max(q, pre);
    if (lane == 0)
      for (int s = 0; s < va.ns && s < armed; ++s) {
        const int last = armed - 1 - ((armed - 1 - s) % va.ns);
        mbar_wait(&bar_full[s], (last / va.ns) & 1, va.err);
      }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int q = 0;
      for (int blk = 0; blk < nblk && ok; ++blk) {
        if (blk >= 1 && !wait(&bar_d_empty, (blk - 1) & 1)) break;
        tc_fence_after();
        for (int c = 0; c < kChunks; ++c, ++q) {
          const int s = q % va.ns;
          if (!wait(&bar_full[s], (q / va.ns) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t wa = smem_u32(smem + s * va.stage_bytes);
          const uint32_t ba = wa + kWChunk;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_desc_sw128(wa + kk * 2048, kWChunk / 2, 1024);
            for (int n0 = 0; n0 < va.bn; n0 += 256) {
              const int n = min(256, va.bn - n0);
              const uint64_t bd = make_desc_sw128(ba + n0 * 128 + kk * 32, 16, 1024);
              umma_ss(tmem + n0, ad, bd, make_idesc_f16(128, n, BF16, true, false),
                      (c | kk) ? 1u : 0u);
            }
          }
          umma_commit(&bar_empty[s]);
        }
        if (ok) umma_commit(&bar_d_full);
      }
      umma_commit(&bar_mma_done);
      mbar_wait(&bar_mma_done, 0, va.err);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------ LSE weights of each row block
    const int wt = threadIdx.x - 64;
    griddep_wait();
    for (int blk = 0; blk < nblk; ++blk) {
      const int b = blk & 1;
      const int t0 = blk * TB;
      const bool ok = blk < 2 || wait_lazy(&bar_wt_empty[b], ((blk >> 1) - 1) & 1);
      if (!named_bar_and(2, 64, ok)) break;
      for (int i = wt; i < np * TB; i += 64) {   // every LSE of the block at once
        const int p = i / TB;
        const int64_t t = t0 + i % TB;
        float v = -INFINITY;
        if (t < va.T)
          v = p < va.P ? __ldg(va.lse_part + (t * va.P + p) * va.H + h)
                       : __ldg(va.lse_local + t * va.H + h);
        s_lse[i] = v;
      }
      named_bar_sync(2, 64);
      for (int t = wt; t < TB; t += 64) {
        float mx = -INFINITY;
        for (int p = 0; p < np; ++p) mx = fmaxf(mx, s_lse[p * TB + t]);
        float sum = 0.f;
        for (int p = 0; p < np; ++p) {
          const float v = s_lse[p * TB + t];
          const float e = (mx == -INFINITY || v == -INFINITY) ? 0.f : __expf(v - mx);
          s_w[b][p * TB + t] = e;
          sum += e;
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        for (int p = 0; p < np; ++p) s_w[b][p * TB + t] *= inv;
        if (va.lse_out && t0 + t < va.T)
          va.lse_out[static_cast<int64_t>(t0 + t) * va.H + h] =
              sum > 0.f ? mx + __logf(sum) : -INFINITY;
      }
      named_bar_sync(2, 64);
      if (wt == 0) mbar_arrive(&bar_wt_full[b]);
    }
  } else {
    // ------------------------------------------------ epilogue (thread = v)
    const int wq = warp & 3;
    const int v = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int nvalid = np * TB;
    uint16_t* o = static_cast<uint16_t*>(va.out);
    griddep_wait();   // an earlier grid may still read out
    for (int blk = 0; blk < nblk; ++blk) {
      const int b = blk & 1;
      const int t0 = blk * TB;
      if (!wait_lazy(&bar_d_full, blk & 1) || !wait_lazy(&bar_wt_full[b], (blk >> 1) & 1)) break;
      tc_fence_after();
      float acc[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] = 0.f;
      const float* w = s_w[b];
      for (int n0 = 0; n0 < nvalid; n0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + n0, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n0 + i < nvalid) {
            // a part of weight 0 (lse = -inf) is skipped, whatever its rows hold
            const float wn = w[n0 + i];
            acc[i % TB] += wn != 0.f ? wn * __uint_as_float(r[i]) : 0.f;
          }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_d_empty);
        mbar_arrive(&bar_wt_empty[b]);
      }
#pragma unroll
      for (int t = 0; t < TB; ++t)
        if (t0 + t < va.T)
          o[(static_cast<int64_t>(t0 + t) * va.H + h) * 128 + v] =
              static_cast<uint16_t>(pack2<BF16>(acc[t], 0.f) & 0xFFFFu);
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, ncols);
  }
}

VupPartsPlan vup_parts_plan(int num_parts, int T) {
  VupPartsPlan pl = {};
  pl.tb = num_parts <= 16 ? 32 : (num_parts <= 32 ? 16 : 8);
  while (pl.tb > 8 && pl.tb / 2 >= T) pl.tb /= 2;
  pl.bn = (num_parts * pl.tb + 15) / 16 * 16;
  pl.stage_bytes = 16384 + pl.bn * 128;
  // static shared memory of the kernel: about 6.3 KB; 1 KB for alignment
  pl.ns = std::min(4, (232448 - 8192 - 1024) / pl.stage_bytes);
  pl.tmem_cols = 32;
  while (pl.tmem_cols < pl.bn) pl.tmem_cols <<= 1;
  pl.smem_bytes = pl.ns * pl.stage_bytes + 1024;
  return pl;
}

template <bool BF16, int TB>
static int launch_vup_parts_t(const CUtensorMap& tm_w, const CUtensorMap& tm_p,
                              const CUtensorMap& tm_l, const VupPartsPlan& plan,
                              const VupPartsArgs& va, cudaStream_t stream) {
  auto kern = mla_vup_parts_kernel<BF16, TB>;
  static int configured[64] = {0};   // largest dynamic shared memory set per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (configured[dev] < plan.smem_bytes) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes) !=
        cudaSuccess)
      return -1;
    configured[dev] = plan.smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(va.H, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_p, tm_l, va) == cudaSuccess ? 0 : -1;
}

int launch_vup_parts(const CUtensorMap& tm_w64, const CUtensorMap& tm_p, const CUtensorMap& tm_l,
                     const VupPartsPlan& plan, bool bf16, int T, int H, int P, bool has_local,
                     const float* lse_part, const float* lse_local, void* out, float* lse_out,
                     int* err, cudaStream_t stream) {
  if (plan.ns < 2 || plan.bn > 512 || P + (has_local ? 1 : 0) > kVupPartsMax) return -1;
  VupPartsArgs va;
  va.T = T;
  va.H = H;
  va.P = P;
  va.has_local = has_local ? 1 : 0;
  va.lse_part = lse_part;
  va.lse_local = lse_local;
  va.out = out;
  va.lse_out = lse_out;
  va.err = err;
  va.ns = plan.ns;
  va.stage_bytes = plan.stage_bytes;
  va.bn = plan.bn;
#define MLA_VP(B, TBV) launch_vup_parts_t<B, TBV>(tm_w64, tm_p, tm_l, plan, va, stream)
  switch (plan.tb) {
    case 32: return bf16 ? MLA_VP(true, 32) : MLA_VP(false, 32);
    case 16: return bf16 ? MLA_VP(true, 16) : MLA_VP(false, 16);
    case 8: return bf16 ? MLA_VP(true, 8) : MLA_VP(false, 8);
    default: return -1;
  }
#undef MLA_VP
}

// ---------------------------------------------------------------- launchers
int launch_combine(const void* o_part, const float* lse_part, int P, const void* o_local,
                   const float* lse_local, int T, int H, int part_dt, int out_dt, void* o_latent,
                   float* lse_out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(T) * H;
  const int blocks = static_cast<int>((rows + 7) / 8);
  if (part_dt == kFP32)
    mla_combine_kernel<true><<<blocks, 256, 0, stream>>>(o_part, lse_part, P, o_local, lse_local, T,
                                                         H, part_dt, out_dt, o_latent, lse_out);
  else
    mla_combine_kernel<false><<<blocks, 256, 0, stream>>>(o_part, lse_part, P, o_local, lse_local,
                                                          T, H, part_dt, out_dt, o_latent, lse_out);
  return 0;
}

int launch_combine_exchanged(const void* o_recv, const float* lse_recv, int nsrc, int P,
                             int hist, int local_src, int T, int H, int part_dt, int out_dt,
                             void* o_latent, float* lse_out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(T) * H;
  const int blocks = static_cast<int>((rows + 7) / 8);
  if (part_dt == kFP32)
    mla_combine_exchanged_kernel<true><<<blocks, 256, 0, stream>>>(
        o_recv, lse_recv, nsrc, P, hist, local_src, T, H, part_dt, out_dt, o_latent, lse_out);
  else
    mla_combine_exchanged_kernel<false><<<blocks, 256, 0, stream>>>(
        o_recv, lse_recv, nsrc, P, hist, local_src, T, H, part_dt, out_dt, o_latent, lse_out);
  return 0;
}

template <bool COMBINE, bool BF16, bool F32>
static int launch_vup_t(const CUtensorMap& tm_w, const void* o_part, const float* lse_part, int P,
                        const void* o_local, const float* lse_local, const void* o_latent_in,
                        int T, int H, int part_dt, void* out, void* o_latent_out, float* lse_out,
                        int* err, cudaStream_t stream) {
  auto kern = mla_vup_kernel<COMBINE, BF16, F32>;
  // the shared-memory limit is a per-device function attribute
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kVupSmem) !=
        cudaSuccess)
      return -1;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = kVupSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tm_w, o_part, lse_part, P, o_local, lse_local, o_latent_in, T,
                         H, part_dt, out, o_latent_out, lse_out, err) != cudaSuccess)
    return -1;
  return 0;
}

int launch_vup(const CUtensorMap& tm_w, bool combine, bool bf16, const void* o_part,
               const float* lse_part, int P, const void* o_local, const float* lse_local,
               const void* o_latent_in, int T, int H, int part_dt, void* out, void* o_latent_out,
               float* lse_out, int* err, cudaStream_t stream) {
#define MLA_VUP_ARGS tm_w, o_part, lse_part, P, o_local, lse_local, o_latent_in, T, H, part_dt, out, \
                     o_latent_out, lse_out, err, stream
  if (!combine)
    return bf16 ? launch_vup_t<false, true, false>(MLA_VUP_ARGS)
                : launch_vup_t<false, false, false>(MLA_VUP_ARGS);
  if (part_dt == kFP32)
    return bf16 ? launch_vup_t<true, true, true>(MLA_VUP_ARGS)
                : launch_vup_t<true, false, true>(MLA_VUP_ARGS);
  return bf16 ? launch_vup_t<true, true, false>(MLA_VUP_ARGS)
              : launch_vup_t<true, false, false>(MLA_VUP_ARGS);
#undef MLA_VUP_ARGS
}

}  // namespace mla
