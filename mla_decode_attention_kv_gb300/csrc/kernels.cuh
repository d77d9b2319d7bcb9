// Launchers of the CUDA kernels and the parameter block of the partial
// kernel, shared by the kernels and the C ABI layer.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mla {

struct PartialParams {
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* o_part;
  float* lse_part;
  int* err;
  int B, q_len, H, num_blocks, bs, max_blocks, S, P, has_cur;
  int T;                 // B * q_len query tokens
  int head_slices;       // o_part / lse_part as [head_slices][T][P][H / head_slices]
  int num_units;
  int box_rows;          // rows per TMA box of the QK CTA's KV maps: min(128, block_size)
  int box_rows_v;        // rows per TMA box of the PV CTA's KV maps: min(64, block_size)
  float scale_log2;      // softmax scale * log2(e) (times kv_scale for an E4M3 cache)
  float out_scale;       // E4M3 cache: kv_scale, applied to O in the epilogue
  uint32_t spin_limit;   // polls before a pipeline wait gives up (MLA_DEV_WAIT_TIMEOUT)
  int part_dtype;        // 0 bf16, 1 fp16, 2 fp32
  // Split-unit workspace (split = number of CTA pairs, 0 = whole units):
  // per pair two slots of O / l and LSE (log2, [128]) for the units cut at
  // the ends of its share, and per pair the record of the split unit whose
  // last tile it holds (+ one header record) and the table of the pairs'
  // share boundaries, read by the merge kernel.
  int split;
  void* ws_o;            // pieces of O / l in the partial dtype, [2*pairs][128][512]
  float* ws_lse;         // [2*pairs][128]
  int4* ws_units;        // [pairs + 1]: {unit, first tile, first pair, last pair}; header {T, pairs}
  int* ws_bounds;        // [pairs + 1]: first tile of each pair's share, then the tile total
};

// Bytes of the workspace's record block: the unit records and the share
// boundaries, rounded up to 256.
inline size_t partial_workspace_recs(int clusters) {
  return (static_cast<size_t>(clusters + 1) * (16 + 4) + 255) / 256 * 256;
}

// Workspace of the partial kernel for `clusters` CTA pairs and partials of
// `part_bytes` bytes per element (4 covers every partial dtype).
inline size_t partial_workspace_bytes(int clusters, int part_bytes = 4) {
  const size_t slots = 2 * static_cast<size_t>(clusters);
  const size_t recs = partial_workspace_recs(clusters);
  return recs + slots * 128 * 4 + slots * 512 * 128 * static_cast<size_t>(part_bytes);
}
int partial_max_clusters();
// Polls before a pipeline wait of the partial kernel gives up: kSpinLimit
// unless a test lowers it (mla_debug_set_spin_limit).
uint32_t partial_spin_limit();

// Rows per TMA box of the partial kernel's KV maps: min(box, block_size) for
// the QK CTA (128-token tiles) and the PV CTA (64-token stages).
constexpr int kPartialBoxK = 128;
constexpr int kPartialBoxV = 64;

int launch_partial(const CUtensorMap& qlat, const CUtensorMap& qpe, const CUtensorMap& kv,
                   const CUtensorMap& cur, const CUtensorMap& kv_v, const CUtensorMap& cur_v,
                   const PartialParams& pp, bool bf16, cudaStream_t stream);
// The partial kernel over an E4M3 cache: kv / cur maps of 128-byte boxes
// (min(128, block_size) rows), kv_v / cur_v of 128-byte boxes of
// min(64, block_size) rows; qlat / qpe as for the 16-bit kernel.
int launch_partial_fp8(const CUtensorMap& qlat, const CUtensorMap& qpe, const CUtensorMap& kv,
                       const CUtensorMap& cur, const CUtensorMap& kv_v, const CUtensorMap& cur_v,
                       const PartialParams& pp, bool bf16, cudaStream_t stream);
int partial_fp8_max_clusters();
// Combine of partials received from an all-to-all: parts (src, p < hist)
// of [nsrc][T][P][H] rows, then part hist of source local_src (if >= 0).
int launch_combine_exchanged(const void* o_recv, const float* lse_recv, int nsrc, int P,
                             int hist, int local_src, int T, int H, int part_dt, int out_dt,
                             void* o_latent, float* lse_out, cudaStream_t stream);
int launch_combine(const void* o_part, const float* lse_part, int P, const void* o_local,
                   const float* lse_local, int T, int H, int part_dt, int out_dt, void* o_latent,
                   float* lse_out, cudaStream_t stream);
int launch_vup(const CUtensorMap& tm_w, bool combine, bool bf16, const void* o_part,
               const float* lse_part, int P, const void* o_local, const float* lse_local,
               const void* o_latent_in, int T, int H, int part_dt, void* out, void* o_latent_out,
               float* lse_out, int* err, cudaStream_t stream);
// mla_lse_combine_vup through the V-up of every part (partials in the
// storage dtype, at most kVupPartsMax parts): the row block and ring plan.
constexpr int kVupPartsMax = 64;
struct VupPartsPlan {
  int tb;            // rows per block: 8, 16 or 32
  int bn;            // B rows per K chunk: parts * tb rounded up to 16
  int stage_bytes;   // W chunk (16 KB) + B chunk
  int ns;            // ring stages
  int tmem_cols;
  int smem_bytes;    // dynamic shared memory
};
VupPartsPlan vup_parts_plan(int num_parts, int T);
int launch_vup_parts(const CUtensorMap& tm_w64, const CUtensorMap& tm_p, const CUtensorMap& tm_l,
                     const VupPartsPlan& plan, bool bf16, int T, int H, int P, bool has_local,
                     const float* lse_part, const float* lse_local, void* out, float* lse_out,
                     int* err, cudaStream_t stream);
int launch_gather(const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                  int B, int num_blocks, int bs, int max_blocks, int max_len, void* dst, int* err,
                  cudaStream_t stream);

}  // namespace mla
