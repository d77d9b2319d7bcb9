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
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

// ---------------------------------------------------------------- weights
// Weights of the parts of row (t, h); returns LSE (natural log) and writes
// the normalised weights (0 for empty parts).  Every lane computes the same
// values in the same order.
__device__ __forceinline__ float combine_weights(const float* lse_part, int P, int H, int64_t t,
                                                 int h, const float* lse_local, float* w) {
  const int np = P + (lse_local ? 1 : 0);
  float mx = -INFINITY;
  for (int p = 0; p < np; ++p) {
    const float v = p < P ? lse_part[(t * P + p) * H + h] : lse_local[t * H + h];
    w[p] = v;
    mx = fmaxf(mx, v);
  }
  if (mx == -INFINITY) {
    for (int p = 0; p < np; ++p) w[p] = 0.f;
    return -INFINITY;
  }
  float sum = 0.f;
  for (int p = 0; p < np; ++p) {
    w[p] = w[p] == -INFINITY ? 0.f : __expf(w[p] - mx);
    sum += w[p];
  }
  const float inv = 1.f / sum;
  for (int p = 0; p < np; ++p) w[p] *= inv;
  return mx + __logf(sum);
}

// Accumulate 16 consecutive elements of one partial row into acc.
__device__ __forceinline__ void accum16(const void* src, int64_t e, int dt, float w,
                                        float (&acc)[16]) {
  if (dt == kFP32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + e);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldg(p + q);
      acc[4 * q] += w * v.x;
      acc[4 * q + 1] += w * v.y;
      acc[4 * q + 2] += w * v.z;
      acc[4 * q + 3] += w * v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + e);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 v = __ldg(p + q);
      const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = unpack2(ws[k], dt);
        acc[8 * q + 2 * k] += w * f.x;
        acc[8 * q + 2 * k + 1] += w * f.y;
      }
    }
  }
}

// Combine row (t, h) for the 16 latent elements of this lane.
__device__ __forceinline__ float combine_row16(const void* o_part, const float* lse_part, int P,
                                               const void* o_local, const float* lse_local,
                                               int H, int64_t t, int h, int part_dt, int lane,
                                               float (&acc)[16]) {
  float w[65];
  const float lse = combine_weights(lse_part, P, H, t, h, lse_local, w);
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int p = 0; p < P; ++p)
    if (w[p] != 0.f) accum16(o_part, ((t * P + p) * H + h) * 512 + lane * 16, part_dt, w[p], acc);
  if (o_local && w[P] != 0.f) accum16(o_local, (t * H + h) * 512 + lane * 16, part_dt, w[P], acc);
  return lse;
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
__global__ void __launch_bounds__(256) mla_combine_kernel(const void* o_part, const float* lse_part,
                                                          int P, const void* o_local,
                                                          const float* lse_local, int T, int H,
                                                          int part_dt, int out_dt, void* o_latent,
                                                          float* lse_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(T) * H) return;
  const int64_t t = row / H;
  const int h = static_cast<int>(row % H);
  float acc[16];
  const float lse =
      combine_row16(o_part, lse_part, P, o_local, lse_local, H, t, h, part_dt, lane, acc);
  store16(o_latent, row * 512 + lane * 16, acc, out_dt);
  if (lse_out && lane == 0) lse_out[row] = lse;
}

// ---------------------------------------------------------------- V-up
constexpr int kVupRows = 64;                    // rows (N) per MMA tile
constexpr int kVupWBytes = 512 * 128 * 2;       // W_UV[h]: 128 KB
constexpr int kVupBBytes = 8 * kVupRows * 128;  // 8 chunks of 64 rows x 128 B: 64 KB
constexpr int kVupSmem = kVupWBytes + kVupBBytes + 1024;

// One CTA per head.  COMBINE: B rows come from the LSE combine of the
// partials; otherwise they are read from o_latent.
template <bool COMBINE, bool BF16>
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
  constexpr uint32_t idesc = make_idesc_f16(128, kVupRows, BF16, true, false);
  bool ok = true;
  int phase = 0;
  for (int t0 = 0; t0 < T && ok; t0 += kVupRows, phase ^= 1) {
    const int nrows = min(kVupRows, T - t0);
    // ---- B operand: rows t0 .. t0 + 63 of head h, latent K-major, SW128
    for (int rr = warp; rr < kVupRows; rr += 8) {
      float acc[16];
      const int64_t t = t0 + rr;
      if (rr < nrows) {
        if constexpr (COMBINE) {
          const float lse = combine_row16(o_part, lse_part, P, o_local, lse_local, H, t, h,
                                          part_dt, lane, acc);
          if (o_latent_out) store16(o_latent_out, (t * H + h) * 512 + lane * 16, acc, dt);
          if (lse_out && lane == 0) lse_out[t * H + h] = lse;
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const uint16_t*>(o_latent_in) + (t * H + h) * 512 + lane * 16);
          const uint4 a = __ldg(src), b = __ldg(src + 1);
          const int c = lane >> 2;
          const int u = 2 * (lane & 3);
          *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u)) = a;
          *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u + 1)) = b;
          continue;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
      }
      const int c = lane >> 2;          // 64-element chunk of this lane's 16 values
      const int u = 2 * (lane & 3);     // first 16-byte unit inside the 128-byte row
      uint32_t wv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) wv[k] = pack2<BF16>(acc[2 * k], acc[2 * k + 1]);
      *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u)) =
          make_uint4(wv[0], wv[1], wv[2], wv[3]);
      *reinterpret_cast<uint4*>(sB + c * (kVupRows * 128) + sw128_offset(rr, u + 1)) =
          make_uint4(wv[4], wv[5], wv[6], wv[7]);
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
      tmem_wait_ld();
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

// ---------------------------------------------------------------- launchers
int launch_combine(const void* o_part, const float* lse_part, int P, const void* o_local,
                   const float* lse_local, int T, int H, int part_dt, int out_dt, void* o_latent,
                   float* lse_out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(T) * H;
  const int blocks = static_cast<int>((rows + 7) / 8);
  mla_combine_kernel<<<blocks, 256, 0, stream>>>(o_part, lse_part, P, o_local, lse_local, T, H,
                                                 part_dt, out_dt, o_latent, lse_out);
  return 0;
}

template <bool COMBINE, bool BF16>
static int launch_vup_t(const CUtensorMap& tm_w, const void* o_part, const float* lse_part, int P,
                        const void* o_local, const float* lse_local, const void* o_latent_in,
                        int T, int H, int part_dt, void* out, void* o_latent_out, float* lse_out,
                        int* err, cudaStream_t stream) {
  auto kern = mla_vup_kernel<COMBINE, BF16>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kVupSmem) !=
        cudaSuccess)
      return -1;
    configured = true;
  }
  kern<<<H, 256, kVupSmem, stream>>>(tm_w, o_part, lse_part, P, o_local, lse_local, o_latent_in,
                                     T, H, part_dt, out, o_latent_out, lse_out, err);
  return 0;
}

int launch_vup(const CUtensorMap& tm_w, bool combine, bool bf16, const void* o_part,
               const float* lse_part, int P, const void* o_local, const float* lse_local,
               const void* o_latent_in, int T, int H, int part_dt, void* out, void* o_latent_out,
               float* lse_out, int* err, cudaStream_t stream) {
  if (combine)
    return bf16 ? launch_vup_t<true, true>(tm_w, o_part, lse_part, P, o_local, lse_local,
                                           o_latent_in, T, H, part_dt, out, o_latent_out, lse_out,
                                           err, stream)
                : launch_vup_t<true, false>(tm_w, o_part, lse_part, P, o_local, lse_local,
                                            o_latent_in, T, H, part_dt, out, o_latent_out,
                                            lse_out, err, stream);
  return bf16 ? launch_vup_t<false, true>(tm_w, o_part, lse_part, P, o_local, lse_local,
                                          o_latent_in, T, H, part_dt, out, o_latent_out, lse_out,
                                          err, stream)
              : launch_vup_t<false, false>(tm_w, o_part, lse_part, P, o_local, lse_local,
                                           o_latent_in, T, H, part_dt, out, o_latent_out, lse_out,
                                           err, stream);
}

}  // namespace mla
