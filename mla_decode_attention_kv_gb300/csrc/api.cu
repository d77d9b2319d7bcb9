// C ABI of the library (declared in include/mla_dcp.h): host-side argument
// checks, TMA tensor-map encoding and kernel launches.  No call allocates
// device memory or synchronises the host.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>
#include "../../include/mla_dcp.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over a row-major [rows, cols] 16-bit tensor, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
              uint32_t box_cols, uint32_t box_rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over [d2, d1, 512] 16-bit elements (row strides in bytes) with a
// box of 64 x 1 x box_d2 and 128-byte swizzle: box_d2 rows of one (d1) slice.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint64_t stride1,
                 uint64_t stride2, uint32_t box_d2, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {512, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {64, 1, box_d2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows, cols] byte tensor (E4M3 values), 128-byte
// swizzle; the part of a box past `cols` is zero-filled.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_half_dtype(int d) { return d == MLA_BF16 || d == MLA_FP16; }
bool is_part_dtype(int d) { return d == MLA_BF16 || d == MLA_FP16 || d == MLA_FP32; }

int launched(int rc) {
  if (rc != 0) return MLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_version(void) { return 100; }

}  // extern "C"

namespace {
std::atomic<uint32_t> g_spin_limit{0};   // 0: the kernels' default
}  // namespace

uint32_t mla::partial_spin_limit() {
  const uint32_t v = g_spin_limit.load(std::memory_order_relaxed);
  return v ? v : mla::kSpinLimit;
}

extern "C" {

void mla_debug_set_spin_limit(uint32_t polls) {
  g_spin_limit.store(polls, std::memory_order_relaxed);
}

const char* mla_get_error_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case MLA_ERR_BAD_SHAPE: return "a size is out of range or inconsistent";
    case MLA_ERR_BAD_DTYPE: return "dtype not supported for this argument";
    case MLA_ERR_MISALIGNED: return "a base pointer is not 16-byte aligned";
    case MLA_ERR_BAD_SHARDS: return "num_shards / num_parts out of range";
    case MLA_ERR_BAD_BLOCK: return "block_size unsupported";
    case MLA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    default: return "unknown status";
  }
}

const char* mla_device_error_string(int code) {
  switch (code) {
    case MLA_DEV_OK: return "ok";
    case MLA_DEV_BAD_BLOCK_ID: return "block_table entry outside [0, num_blocks)";
    case MLA_DEV_WAIT_TIMEOUT: return "a pipeline wait exceeded its spin budget";
    case MLA_DEV_BAD_SEQ_LEN: return "seq_lens entry outside [0, max_blocks * block_size]";
    default: return "unknown device error";
  }
}

}  // extern "C"

namespace {
// Host checks of mla_dcp_decode_partial's arguments (all but the workspace).
int check_partial_args(const void* q_abs, const void* q_pe, const void* kv_cache,
                       const int32_t* block_table, const int32_t* seq_lens, const void* kv_cur,
                       int B, int q_len, int H, int num_blocks, int block_size, int max_blocks,
                       int num_shards, float scale, int in_dtype, int part_dtype,
                       const void* o_part, const float* lse_part) {
  if (!q_abs || !q_pe || !kv_cache || !block_table || !seq_lens || !o_part || !lse_part)
    return MLA_ERR_NULL_POINTER;
  if (!is_half_dtype(in_dtype) || !is_part_dtype(part_dtype)) return MLA_ERR_BAD_DTYPE;
  if (B < 1 || q_len < 1 || q_len > MLA_MAX_Q_LEN || H < 1 || H > MLA_MAX_HEADS || num_blocks < 1 ||
      max_blocks < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return MLA_ERR_BAD_SHAPE;
  if (num_shards < 1 || num_shards > MLA_MAX_SHARDS) return MLA_ERR_BAD_SHARDS;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128 &&
      block_size != 256)
    return MLA_ERR_BAD_BLOCK;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX ||
      static_cast<int64_t>(B) * q_len * H > INT32_MAX / 2)
    return MLA_ERR_BAD_SHAPE;
  if (!aligned16(q_abs) || !aligned16(q_pe) || !aligned16(kv_cache) || !aligned16(o_part) ||
      (kv_cur && !aligned16(kv_cur)) || !aligned16(lse_part))
    return MLA_ERR_MISALIGNED;
  if (static_cast<int64_t>(B) * q_len * (num_shards + (kv_cur ? 1 : 0)) > INT32_MAX)
    return MLA_ERR_BAD_SHAPE;
  return MLA_OK;
}
}  // namespace

namespace {
// The partial call over a 16-bit cache (kv8 false: kv values in in_dtype) or
// an E4M3 cache (kv8 true: one byte per value, times kv_scale).
int decode_partial(bool kv8, const void* q_abs, const void* q_pe, const void* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const void* kv_cur, int B,
                   int q_len, int H, int num_blocks, int block_size, int max_blocks,
                   int num_shards, float scale, float kv_scale, int in_dtype, int part_dtype,
                   void* o_part, float* lse_part, int32_t* err_flag, void* workspace,
                   uint64_t workspace_bytes, int head_slices, mla_stream_t stream) {
  const int rc = check_partial_args(q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B,
                                    q_len, H, num_blocks, block_size, max_blocks, num_shards,
                                    scale, in_dtype, part_dtype, o_part, lse_part);
  if (rc != MLA_OK) return rc;
  if (kv8 && (!(kv_scale > 0.f) || !std::isfinite(kv_scale) ||
              !std::isfinite(scale * kv_scale * 1.4426950408889634f)))
    return MLA_ERR_BAD_SHAPE;
  if (head_slices < 1 || H % head_slices != 0) return MLA_ERR_BAD_SHAPE;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MLA_ERR_MISALIGNED;

  const bool bf16 = in_dtype == MLA_BF16;
  const int box_k = block_size < mla::kPartialBoxK ? block_size : mla::kPartialBoxK;
  const int box_v = block_size < mla::kPartialBoxV ? block_size : mla::kPartialBoxV;
  const uint64_t qrows = static_cast<uint64_t>(B) * q_len * H;
  const uint64_t kv_rows = static_cast<uint64_t>(num_blocks) * block_size;
  const uint64_t cur_rows = static_cast<uint64_t>(B) * q_len;
  CUtensorMap tm_qlat, tm_qpe, tm_kv, tm_cur, tm_kv_v, tm_cur_v;
  if (!make_map(&tm_qlat, q_abs, 512, qrows, 1024, 64, 128, bf16) ||
      !make_map(&tm_qpe, q_pe, 64, qrows, 128, 64, 128, bf16))
    return MLA_ERR_CUDA;
  if (kv8) {
    // 576-byte token rows in 128-byte boxes
    if (!make_map_u8(&tm_kv, kv_cache, 576, kv_rows, 576, 128, box_k) ||
        !make_map_u8(&tm_kv_v, kv_cache, 576, kv_rows, 576, 128, box_v) ||
        (kv_cur && (!make_map_u8(&tm_cur, kv_cur, 576, cur_rows, 576, 128, box_k) ||
                    !make_map_u8(&tm_cur_v, kv_cur, 576, cur_rows, 576, 128, box_v))))
      return MLA_ERR_CUDA;
  } else {
    if (!make_map(&tm_kv, kv_cache, 576, kv_rows, 1152, 64, box_k, bf16) ||
        !make_map(&tm_kv_v, kv_cache, 576, kv_rows, 1152, 64, box_v, bf16) ||
        (kv_cur && (!make_map(&tm_cur, kv_cur, 576, cur_rows, 1152, 64, box_k, bf16) ||
                    !make_map(&tm_cur_v, kv_cur, 576, cur_rows, 1152, 64, box_v, bf16))))
      return MLA_ERR_CUDA;
  }
  if (!kv_cur) {
    tm_cur = tm_kv;     // never read
    tm_cur_v = tm_kv_v;
  }

  mla::PartialParams pp;
  pp.block_table = block_table;
  pp.seq_lens = seq_lens;
  pp.o_part = o_part;
  pp.lse_part = lse_part;
  pp.err = err_flag;
  pp.B = B;
  pp.q_len = q_len;
  pp.H = H;
  pp.num_blocks = num_blocks;
  pp.bs = block_size;
  pp.max_blocks = max_blocks;
  pp.S = num_shards;
  pp.has_cur = kv_cur ? 1 : 0;
  pp.P = num_shards + pp.has_cur;
  pp.num_units = B * q_len * pp.P;   // checked above to fit an int
  pp.T = B * q_len;
  pp.head_slices = head_slices;
  pp.box_rows = box_k;
  pp.box_rows_v = box_v;
  pp.scale_log2 = scale * (kv8 ? kv_scale : 1.f) * 1.4426950408889634f;
  pp.out_scale = kv8 ? kv_scale : 1.f;
  pp.spin_limit = mla::partial_spin_limit();
  pp.part_dtype = part_dtype;
  pp.split = 0;
  pp.ws_o = nullptr;
  pp.ws_lse = nullptr;
  pp.ws_units = nullptr;
  pp.ws_bounds = nullptr;
  if (workspace) {
    const int clusters = mla::partial_max_clusters();
    if (clusters < 1) return MLA_ERR_CUDA;
    const int part_bytes = part_dtype == MLA_FP32 ? 4 : 2;
    if (workspace_bytes < mla::partial_workspace_bytes(clusters, part_bytes)) return MLA_ERR_BAD_SHAPE;
    const size_t recs = mla::partial_workspace_recs(clusters);
    char* w = static_cast<char*>(workspace);
    pp.split = clusters;
    pp.ws_units = reinterpret_cast<int4*>(w);
    pp.ws_bounds = reinterpret_cast<int*>(w + static_cast<size_t>(clusters + 1) * 16);
    pp.ws_lse = reinterpret_cast<float*>(w + recs);
    pp.ws_o = w + recs + 2 * static_cast<size_t>(clusters) * 128 * 4;
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launched(kv8 ? mla::launch_partial_fp8(tm_qlat, tm_qpe, tm_kv, tm_cur, tm_kv_v, tm_cur_v,
                                                pp, bf16, st)
                      : mla::launch_partial(tm_qlat, tm_qpe, tm_kv, tm_cur, tm_kv_v, tm_cur_v, pp,
                                            bf16, st));
}
}  // namespace

extern "C" {

int mla_dcp_decode_partial_sliced(const void* q_abs, const void* q_pe, const void* kv_cache,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const void* kv_cur, int B, int q_len, int H, int num_blocks,
                                  int block_size, int max_blocks, int num_shards, float scale,
                                  int in_dtype, int part_dtype, void* o_part, float* lse_part,
                                  int32_t* err_flag, void* workspace, uint64_t workspace_bytes,
                                  int head_slices, mla_stream_t stream) {
  return decode_partial(false, q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B, q_len, H,
                        num_blocks, block_size, max_blocks, num_shards, scale, 1.f, in_dtype,
                        part_dtype, o_part, lse_part, err_flag, workspace, workspace_bytes,
                        head_slices, stream);
}

int mla_dcp_decode_partial_fp8(const void* q_abs, const void* q_pe, const void* kv_cache,
                               const int32_t* block_table, const int32_t* seq_lens,
                               const void* kv_cur, int B, int q_len, int H, int num_blocks,
                               int block_size, int max_blocks, int num_shards, float scale,
                               float kv_scale, int in_dtype, int part_dtype, void* o_part,
                               float* lse_part, int32_t* err_flag, void* workspace,
                               uint64_t workspace_bytes, int head_slices, mla_stream_t stream) {
  return decode_partial(true, q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B, q_len, H,
                        num_blocks, block_size, max_blocks, num_shards, scale, kv_scale, in_dtype,
                        part_dtype, o_part, lse_part, err_flag, workspace, workspace_bytes,
                        head_slices, stream);
}

int mla_dcp_decode_partial(const void* q_abs, const void* q_pe, const void* kv_cache,
                           const int32_t* block_table, const int32_t* seq_lens,
                           const void* kv_cur, int B, int q_len, int H, int num_blocks,
                           int block_size, int max_blocks, int num_shards, float scale,
                           int in_dtype, int part_dtype, void* o_part, float* lse_part,
                           int32_t* err_flag, void* workspace, uint64_t workspace_bytes,
                           mla_stream_t stream) {
  return mla_dcp_decode_partial_sliced(q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B,
                                       q_len, H, num_blocks, block_size, max_blocks, num_shards,
                                       scale, in_dtype, part_dtype, o_part, lse_part, err_flag,
                                       workspace, workspace_bytes, 1, stream);
}

uint64_t mla_dcp_decode_partial_workspace_size(int B, int q_len, int num_shards, int has_current) {
  if (B < 1 || q_len < 1 || q_len > MLA_MAX_Q_LEN || num_shards < 1 || num_shards > MLA_MAX_SHARDS) return 0;
  const int64_t units = static_cast<int64_t>(B) * q_len * (num_shards + (has_current ? 1 : 0));
  if (units > INT32_MAX) return 0;
  const int clusters = mla::partial_max_clusters();
  if (clusters < 1) return 0;
  return mla::partial_workspace_bytes(clusters);
}

// ------------------------------------------------------------------ no-alloc variant
// Scratch of mla_dcp_decode_partial_noalloc: a fixed device array, so the
// call needs no allocation of any kind.  24 MiB holds the split-shard
// workspace of up to 95 CTA pairs with 16-bit partials (47 with fp32).
constexpr size_t kNoAllocScratchBytes = size_t{24} << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_noalloc_scratch, looked up once per device with that
// device current, and again if the device's context changed since (after a
// cudaDeviceReset the array lives in a new context, at a new address).
void* noalloc_scratch() {
  static void* addr[64] = {nullptr};
  static CUcontext owner[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return nullptr;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;   // null before the first runtime call
  std::lock_guard<std::mutex> lock(mu);
  if (!ctx || !addr[dev] || owner[dev] != ctx) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess) {   // sets up the context
      cudaGetLastError();
      return nullptr;
    }
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    addr[dev] = a;
    owner[dev] = ctx;
  }
  return addr[dev];
}
}  // namespace

int mla_dcp_decode_partial_noalloc(const void* q_abs, const void* q_pe, const void* kv_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const void* kv_cur, int B, int q_len, int H, int num_blocks,
                                   int block_size, int max_blocks, int num_shards, float scale,
                                   int in_dtype, int part_dtype, void* o_part, float* lse_part,
                                   int32_t* err_flag, mla_stream_t stream) {
  // the same argument checks, in the same order, as the workspace entry point
  const int rc = check_partial_args(q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B,
                                    q_len, H, num_blocks, block_size, max_blocks, num_shards,
                                    scale, in_dtype, part_dtype, o_part, lse_part);
  if (rc != MLA_OK) return rc;
  const int clusters = mla::partial_max_clusters();
  if (clusters < 1) return MLA_ERR_CUDA;
  const size_t need = mla::partial_workspace_bytes(clusters, part_dtype == MLA_FP32 ? 4 : 2);
  void* scratch = nullptr;
  if (need <= kNoAllocScratchBytes) {
    scratch = noalloc_scratch();
    if (!scratch) return MLA_ERR_CUDA;
  }
  // when the split-shard scratch of this device's pairs does not fit the
  // array (fp32 partials on a GPU with more than 47 pairs), every pair takes
  // whole shards instead: the same results, with no scratch at all
  return mla_dcp_decode_partial(q_abs, q_pe, kv_cache, block_table, seq_lens, kv_cur, B, q_len, H,
                                num_blocks, block_size, max_blocks, num_shards, scale, in_dtype,
                                part_dtype, o_part, lse_part, err_flag, scratch,
                                scratch ? need : 0, stream);
}

int mla_lse_combine(const void* o_part, const float* lse_part, int num_parts, const void* o_local,
                    const float* lse_local, int T, int H, int part_dtype, int out_dtype,
                    void* o_latent, float* lse_out, mla_stream_t stream) {
  if (!o_part || !lse_part || !o_latent) return MLA_ERR_NULL_POINTER;
  if ((o_local == nullptr) != (lse_local == nullptr)) return MLA_ERR_NULL_POINTER;
  if (!is_part_dtype(part_dtype) || !is_part_dtype(out_dtype)) return MLA_ERR_BAD_DTYPE;
  if (T < 1 || H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_BAD_SHAPE;
  if (num_parts < 1 || num_parts > MLA_MAX_SHARDS + 1) return MLA_ERR_BAD_SHARDS;
  if (!aligned16(o_part) || !aligned16(o_latent) || (o_local && !aligned16(o_local)))
    return MLA_ERR_MISALIGNED;
  return launched(mla::launch_combine(o_part, lse_part, num_parts, o_local, lse_local, T, H,
                                      part_dtype, out_dtype, o_latent, lse_out,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int mla_dcp_combine_exchanged(const void* o_recv, const float* lse_recv, int num_src,
                              int parts_per_src, int hist_parts, int local_src, int T, int H,
                              int part_dtype, int out_dtype, void* o_latent, float* lse_out,
                              mla_stream_t stream) {
  if (!o_recv || !lse_recv || !o_latent) return MLA_ERR_NULL_POINTER;
  if (!is_part_dtype(part_dtype) || !is_part_dtype(out_dtype)) return MLA_ERR_BAD_DTYPE;
  if (T < 1 || H < 1 || H > MLA_MAX_HEADS || num_src < 1) return MLA_ERR_BAD_SHAPE;
  if (static_cast<int64_t>(num_src) * T * parts_per_src * H > INT32_MAX / 2)
    return MLA_ERR_BAD_SHAPE;
  if (parts_per_src < 1 || parts_per_src > MLA_MAX_SHARDS + 1 || hist_parts < 0 ||
      hist_parts > parts_per_src || local_src < -1 || local_src >= num_src ||
      (local_src >= 0 && hist_parts >= parts_per_src))
    return MLA_ERR_BAD_SHARDS;
  const int64_t np = static_cast<int64_t>(num_src) * hist_parts + (local_src >= 0 ? 1 : 0);
  if (np < 1 || np > 96) return MLA_ERR_BAD_SHARDS;
  if (!aligned16(o_recv) || !aligned16(o_latent)) return MLA_ERR_MISALIGNED;
  return launched(mla::launch_combine_exchanged(o_recv, lse_recv, num_src, parts_per_src,
                                                hist_parts, local_src, T, H, part_dtype,
                                                out_dtype, o_latent, lse_out,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

static int vup_common(bool combine, const void* o_part, const float* lse_part, int num_parts,
                      const void* o_local, const float* lse_local, const void* o_latent_in,
                      const void* W_UV, int T, int H, int part_dtype, int dtype, void* out,
                      void* o_latent_out, float* lse_out, int32_t* err_flag,
                      mla_stream_t stream) {
  if (!W_UV || !out) return MLA_ERR_NULL_POINTER;
  if (!is_half_dtype(dtype)) return MLA_ERR_BAD_DTYPE;
  if (T < 1 || T > 65536 || H < 1 || H > MLA_MAX_HEADS) return MLA_ERR_BAD_SHAPE;
  if (!aligned16(W_UV) || !aligned16(out)) return MLA_ERR_MISALIGNED;
  const bool bf16 = dtype == MLA_BF16;
  const int nparts = num_parts + (o_local ? 1 : 0);
  if (combine && part_dtype == dtype && nparts <= mla::kVupPartsMax && !o_latent_out) {
    // partials in W_UV's dtype: the V-up of every part, then the weighted sum
    const mla::VupPartsPlan plan = mla::vup_parts_plan(nparts, T);
    const uint64_t row = 1024;   // one 512-element latent row
    CUtensorMap tm_w64, tm_p, tm_l;
    if (!make_map(&tm_w64, W_UV, 128, static_cast<uint64_t>(H) * 512, 256, 64, 64, bf16) ||
        !make_map_3d(&tm_p, o_part, static_cast<uint64_t>(num_parts) * H, T, row,
                     row * num_parts * H, plan.tb, bf16) ||
        !make_map_3d(&tm_l, o_local ? o_local : o_part, H, T, row, row * H, plan.tb, bf16))
      return MLA_ERR_CUDA;
    return launched(mla::launch_vup_parts(tm_w64, tm_p, tm_l, plan, bf16, T, H, num_parts,
                                          o_local != nullptr, lse_part, lse_local, out, lse_out,
                                          err_flag, reinterpret_cast<cudaStream_t>(stream)));
  }
  CUtensorMap tm_w;
  if (!make_map(&tm_w, W_UV, 128, static_cast<uint64_t>(H) * 512, 256, 64, 256, bf16))
    return MLA_ERR_CUDA;
  return launched(mla::launch_vup(tm_w, combine, bf16, o_part, lse_part, num_parts, o_local,
                                  lse_local, o_latent_in, T, H, part_dtype, out, o_latent_out,
                                  lse_out, err_flag, reinterpret_cast<cudaStream_t>(stream)));
}

int mla_vup(const void* o_latent, const void* W_UV, int T, int H, int dtype, void* out,
            int32_t* err_flag, mla_stream_t stream) {
  if (!o_latent) return MLA_ERR_NULL_POINTER;
  if (!aligned16(o_latent)) return MLA_ERR_MISALIGNED;
  return vup_common(false, nullptr, nullptr, 0, nullptr, nullptr, o_latent, W_UV, T, H, dtype,
                    dtype, out, nullptr, nullptr, err_flag, stream);
}

int mla_lse_combine_vup(const void* o_part, const float* lse_part, int num_parts,
                        const void* o_local, const float* lse_local, const void* W_UV, int T,
                        int H, int part_dtype, int dtype, void* out, void* o_latent,
                        float* lse_out, int32_t* err_flag, mla_stream_t stream) {
  if (!o_part || !lse_part) return MLA_ERR_NULL_POINTER;
  if ((o_local == nullptr) != (lse_local == nullptr)) return MLA_ERR_NULL_POINTER;
  if (!is_part_dtype(part_dtype)) return MLA_ERR_BAD_DTYPE;
  if (num_parts < 1 || num_parts > MLA_MAX_SHARDS + 1) return MLA_ERR_BAD_SHARDS;
  if (!aligned16(o_part) || (o_local && !aligned16(o_local)) ||
      (o_latent && !aligned16(o_latent)))
    return MLA_ERR_MISALIGNED;
  return vup_common(true, o_part, lse_part, num_parts, o_local, lse_local, nullptr, W_UV, T, H,
                    part_dtype, dtype, out, o_latent, lse_out, err_flag, stream);
}

int mla_gather_kv(const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens, int B,
                  int num_blocks, int block_size, int max_blocks, int max_len, void* dst,
                  int32_t* err_flag, mla_stream_t stream) {
  if (!kv_cache || !block_table || !seq_lens || !dst) return MLA_ERR_NULL_POINTER;
  if (B < 1 || B > 65535 || num_blocks < 1 || block_size < 1 || max_blocks < 1 || max_len < 1)
    return MLA_ERR_BAD_SHAPE;
  if (!aligned16(kv_cache) || !aligned16(dst)) return MLA_ERR_MISALIGNED;
  return launched(mla::launch_gather(kv_cache, block_table, seq_lens, B, num_blocks, block_size,
                                     max_blocks, max_len, dst, err_flag,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
