// Test hook mla_gather_kv: bit-exact copy of each sequence's paged history
// into a dense buffer.  It follows the HISTORY attention call of the
// vllm-ascend PR #16977 study page (code block B): the cache is read through
// block_table, block_size and the per-sequence history length.
//   dst[b, t, :] = kv_cache[block_table[b][t / bs]][t % bs][:]   (t < L_b)
// Rows t >= L_b are zeroed; an out-of-range block id sets the device error
// word and zeroes its rows.
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

// One warp per token row of 576 x 2 bytes = 72 units of 16 bytes.
__global__ void __launch_bounds__(256) mla_gather_kernel(const uint4* kv_cache,
                                                         const int32_t* block_table,
                                                         const int32_t* seq_lens, int num_blocks,
                                                         int bs, int max_blocks, int max_len,
                                                         uint4* dst, int* err) {
  const int b = blockIdx.y;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= max_len) return;
  constexpr int kUnits = 576 * 2 / 16;
  uint4* out = dst + (static_cast<int64_t>(b) * max_len + t) * kUnits;
  const int L = seq_lens[b];
  if ((L < 0 || L > max_blocks * bs) && t == 0 && lane == 0) set_error(err, kDevBadSeqLen);
  bool valid = t < L && t < max_blocks * bs;
  int64_t src_row = 0;
  if (valid) {
    const int pb = block_table[static_cast<int64_t>(b) * max_blocks + t / bs];
    if (pb < 0 || pb >= num_blocks) {
      if (lane == 0) set_error(err, kDevBadBlockId);
      valid = false;
    } else {
      src_row = static_cast<int64_t>(pb) * bs + t % bs;
    }
  }
  const uint4* src = kv_cache + src_row * kUnits;
  for (int u = lane; u < kUnits; u += 32) out[u] = valid ? src[u] : make_uint4(0, 0, 0, 0);
}

int launch_gather(const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                  int B, int num_blocks, int bs, int max_blocks, int max_len, void* dst, int* err,
                  cudaStream_t stream) {
  dim3 grid((max_len + 7) / 8, B);
  mla_gather_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(kv_cache), block_table,
                                              seq_lens, num_blocks, bs, max_blocks, max_len,
                                              static_cast<uint4*>(dst), err);
  return 0;
}

}  // namespace mla
