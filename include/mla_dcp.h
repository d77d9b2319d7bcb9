/*
 * mla_dcp.h -- C ABI of the GB300 (sm_103a) decode-step MLA library.
 *
 * One decode step of Multi-head Latent Attention over a paged, compressed
 * latent KV cache whose history is split into context shards:
 *
 *   mla_dcp_decode_partial  per-shard (and CURRENT-chunk) partial attention
 *                           outputs and their log-sum-exp
 *   mla_dcp_decode_partial_fp8  the same over an FP8 (E4M3) latent cache
 *   mla_lse_combine         LSE-weighted merge of the partials: the result
 *                           equals one softmax over the whole sequence
 *   mla_vup                 per-head V up-projection, latent 512 -> 128
 *   mla_lse_combine_vup     the combine with the V-up fused into its epilogue
 *   mla_gather_kv           test hook: bit-exact gather of paged history
 *
 * Sources (web pages, cited by title and section):
 *   [PR]  vllm-ascend PR #16977 study page, "DCP decode: streams and V-up"
 *         (huashanblogllm.xyz study-dcp-decode-streams-vup)
 *   [TP]  MLA multi-GPU TP configuration article (hncyxsy.com news 238223)
 *   [K3]  "RTPLLM推理优化：K3芯片上MLA注意力的DCP与通算融合实践" (zwxr.cn 254603)
 *   [KM]  the Kthena x Mooncake KV-cache reuse article (its KV compression
 *         sections 3.2 and 5.2)
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no device memory in any of these calls.
 *   - Tensors are dense, C-contiguous, in the layouts stated per argument.
 *     Every base pointer must be 16-byte aligned.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *     and never synchronises the host.
 *   - Return value: MLA_OK (0) or an mla_status code for errors the host can
 *     see (null pointer, bad size, bad dtype, misalignment, launch failure).
 *     Nothing is launched when a host check fails.
 *   - Errors only the device can see (a block_table entry outside
 *     [0, num_blocks), a seq_lens entry outside [0, max_blocks*block_size],
 *     a pipeline wait that ran out of its spin budget) are
 *     written to *err_flag (a caller-owned device int32, may be NULL) with
 *     the first writer winning; read it after synchronising.  When it is
 *     non-zero the outputs of that call are unspecified.  No kernel traps or
 *     spins without bound.
 */
#ifndef MLA_DCP_H
#define MLA_DCP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* mla_stream_t;

/* Element types.  Q, the cache, kv_cur and W_UV share one storage dtype
 * (BF16 or FP16); partial outputs may also be FP32. */
typedef enum { MLA_BF16 = 0, MLA_FP16 = 1, MLA_FP32 = 2 } mla_dtype;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_NULL_POINTER = 1,  /* a required pointer is NULL                   */
  MLA_ERR_BAD_SHAPE = 2,     /* a size is out of range or inconsistent       */
  MLA_ERR_BAD_DTYPE = 3,     /* dtype not supported for this argument        */
  MLA_ERR_MISALIGNED = 4,    /* a base pointer is not 16-byte aligned        */
  MLA_ERR_BAD_SHARDS = 5,    /* num_shards / num_parts out of range          */
  MLA_ERR_BAD_BLOCK = 6,     /* block_size unsupported                       */
  MLA_ERR_CUDA = 7,          /* a CUDA runtime/driver call failed            */
} mla_status;

/* Device error codes written to *err_flag. */
enum {
  MLA_DEV_OK = 0,
  MLA_DEV_BAD_BLOCK_ID = 1,  /* a block_table entry outside [0, num_blocks)       */
  MLA_DEV_WAIT_TIMEOUT = 2,  /* a pipeline wait ran out of its spin budget         */
  MLA_DEV_BAD_SEQ_LEN = 3    /* a seq_lens entry outside [0, max_blocks*block_size] */
};

enum {
  MLA_D_LATENT = 512, /* kv_lora_rank: width of c_KV  ([TP] "物理矛盾")          */
  MLA_D_ROPE = 64,    /* width of the decoupled RoPE key k_R ([TP] "物理矛盾")   */
  MLA_D_QK = 576,     /* values per cached token ([TP] route A, ~1.15 KB/token) */
  MLA_D_V = 128,      /* per-head V width after the up-projection ([PR] block A) */
  MLA_MAX_HEADS = 128,
  MLA_MAX_SHARDS = 64,
  /* query tokens per sequence: decode (1), MTP (2) and CURRENT chunks of a
   * chunked prefill up to 64 ([PR] closing paragraph of the proposal keeps
   * prefill itself on the old path); the CURRENT part of query i covers
   * kv_cur[b, 0..i], one KV tile of the partial kernel */
  MLA_MAX_Q_LEN = 64
};

/*
 * mla_dcp_decode_partial -- partial attention per context shard.
 *
 * Defines: [PR] glossary "DCP" and "LSE", and the HISTORY / CURRENT split of
 * the decode step (the section on the two-segment decode step; code blocks B and C):
 * the history KV is split along the sequence into `num_shards` shards, each
 * shard yields a partial output and its LSE; the CURRENT chunk is attended
 * with a causal window mask and yields one more partial.
 *
 * For sequence b, query token i, head h and part p:
 *   s_t   = scale * (q_abs[b,i,h,:] . c_t + q_pe[b,i,h,:] . kR_t)
 *   o_part[b,i,p,h,:] = sum_t softmax_t(s) * c_t   over the part's tokens
 *   lse_part[b,i,p,h] = ln sum_t exp(s_t)          (natural log)
 * where c_t = cache entry [0:512) and kR_t = [512:576).  History token t of
 * sequence b is kv_cache[block_table[b][t / block_size]][t % block_size].
 * Shard s (0 <= s < num_shards) covers history tokens
 *   [s*len, min(L_b, (s+1)*len)),  len = block_size * ceil(L_b / (num_shards*block_size)),
 * L_b = seq_lens[b].  History is fully visible to every query token.
 * If kv_cur != NULL, part p = num_shards is the CURRENT segment: query token
 * i sees kv_cur[b, j] for j <= i.
 * A part with no visible token gets o = 0 and lse = -inf.
 *
 * Arguments
 *   q_abs      [B, q_len, H, 512] in_dtype  query absorbed into latent space
 *   q_pe       [B, q_len, H, 64]  in_dtype  RoPE query, already rotated
 *   kv_cache   [num_blocks, block_size, 576] in_dtype.  The slots of a
 *              sequence's last block past L_b are read with the block (and
 *              weighted by 0), so they must hold finite values.
 *   block_table[B, max_blocks] int32   physical block ids; entries past
 *              ceil(L_b / block_size) are never read
 *   seq_lens   [B] int32 (device)  history lengths, 0 <= L_b <= max_blocks*block_size;
 *              an entry outside that range sets MLA_DEV_BAD_SEQ_LEN
 *   kv_cur     [B, q_len, 576] in_dtype, or NULL (no CURRENT segment)
 *   B >= 1; 1 <= q_len <= 64; 1 <= H <= 128; block_size in {16,32,64,128,256};
 *   1 <= num_shards <= 64; scale > 0 (1/sqrt(192) for the 128+64 head width)
 *   in_dtype   MLA_BF16 or MLA_FP16;  part_dtype MLA_BF16, MLA_FP16 or MLA_FP32
 *   o_part     [B, q_len, P, H, 512] part_dtype, P = num_shards + (kv_cur != NULL)
 *   lse_part   [B, q_len, P, H] float32
 *   err_flag   device int32 or NULL (see conventions)
 *   workspace  device scratch of at least workspace_bytes, or NULL; needs
 *              no initialisation.  With a workspace the GPU's CTA pairs take
 *              equal shares of the work (every KV tile, plus half a tile's
 *              worth per shard piece) whenever whole shards would leave them
 *              uneven; a shard cut between pairs has its pieces parked there
 *              and merged by their LSEs (as in mla_lse_combine) into o_part /
 *              lse_part by a second kernel on the same stream.  Without one
 *              each pair takes whole shards.
 *              Calls that may overlap in time need separate workspaces.
 *   workspace_bytes  size of workspace; at least
 *              mla_dcp_decode_partial_workspace_size(B, q_len, num_shards,
 *              kv_cur != NULL) when workspace != NULL.
 * Returns MLA_OK or an mla_status.
 */
int mla_dcp_decode_partial(const void* q_abs, const void* q_pe, const void* kv_cache,
                           const int32_t* block_table, const int32_t* seq_lens,
                           const void* kv_cur, int B, int q_len, int H, int num_blocks,
                           int block_size, int max_blocks, int num_shards, float scale,
                           int in_dtype, int part_dtype, void* o_part, float* lse_part,
                           int32_t* err_flag, void* workspace, uint64_t workspace_bytes,
                           mla_stream_t stream);

/*
 * mla_dcp_decode_partial_sliced -- mla_dcp_decode_partial with its partials
 * laid out for an exchange between GPUs that scatters heads.
 *
 * Defines: [PR] the third change (the HISTORY partials of every rank go
 * through one all-to-all with scatter_dim = 1, the heads, before the
 * combine).  With head_slices = N (dividing H), o_part is
 * [N][B*q_len][P][H/N][512] and lse_part [N][B*q_len][P][H/N]: head h of
 * token t = b*q_len + i, part p is row ((h / (H/N)) * B*q_len + t) * P + p)
 * * (H/N) + h % (H/N).  Block n (heads [n*H/N, (n+1)*H/N)) is contiguous,
 * so it is exactly what rank n receives from an all-to-all of equal
 * splits.  head_slices = 1 is mla_dcp_decode_partial.  Every other argument,
 * result and error as mla_dcp_decode_partial; MLA_ERR_BAD_SHAPE if
 * head_slices < 1 or does not divide H.
 */
int mla_dcp_decode_partial_sliced(const void* q_abs, const void* q_pe, const void* kv_cache,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const void* kv_cur, int B, int q_len, int H, int num_blocks,
                                  int block_size, int max_blocks, int num_shards, float scale,
                                  int in_dtype, int part_dtype, void* o_part, float* lse_part,
                                  int32_t* err_flag, void* workspace, uint64_t workspace_bytes,
                                  int head_slices, mla_stream_t stream);

/*
 * mla_dcp_decode_partial_fp8 -- mla_dcp_decode_partial_sliced over an FP8
 * latent cache.
 *
 * Defines: the KV compression direction of [KM] (sections 3.2 and 5.2),
 * which the sources only point towards; the format is this library's
 * reading: every cached value, history and CURRENT, latent and RoPE, is one
 * E4M3 byte e (OCP FP8: bias 7, 3 mantissa bits, no infinities, 0x7F / 0xFF
 * NaN) times one per-tensor kv_scale, so that c_t and kR_t above are the
 * decoded bytes times kv_scale.  The results are those of
 * mla_dcp_decode_partial on those values.
 *
 * Differences from mla_dcp_decode_partial_sliced:
 *   kv_cache   [num_blocks, block_size, 576] bytes (E4M3); as for the 16-bit
 *              cache, the slots of a last block past L_b are read with the
 *              block and weighted by 0, so they must not hold the NaN codes
 *   kv_cur     [B, q_len, 576] bytes (E4M3, the same kv_scale), or NULL
 *   kv_scale   > 0 and finite (scale * kv_scale too); MLA_ERR_BAD_SHAPE otherwise
 * Precision: the tensor cores multiply the cache bytes by the query in two
 * E4M3 terms (a power-of-two row scale, then the rounded row and its rounded
 * remainder), which keeps |error of q| <= 2^-8 |q| + 2^-17 max|q row|,
 * about the precision of bf16; the softmax weights p (at most 4 times the
 * running maximum) go to the PV product in the same two-term form of 2^6 p
 * (rounded to fp16 first): |error of p| <= 2^-7 p + 2^-16.  Every other argument, result and error
 * (including the workspace, of the same size) as
 * mla_dcp_decode_partial_sliced.
 */
int mla_dcp_decode_partial_fp8(const void* q_abs, const void* q_pe, const void* kv_cache,
                               const int32_t* block_table, const int32_t* seq_lens,
                               const void* kv_cur, int B, int q_len, int H, int num_blocks,
                               int block_size, int max_blocks, int num_shards, float scale,
                               float kv_scale, int in_dtype, int part_dtype, void* o_part,
                               float* lse_part, int32_t* err_flag, void* workspace,
                               uint64_t workspace_bytes, int head_slices, mla_stream_t stream);

/*
 * mla_dcp_decode_partial_workspace_size -- bytes of workspace that
 * mla_dcp_decode_partial needs on the current device: about 0.5 MiB per
 * CTA pair the device keeps resident (FP32 partials need twice that), with
 * no term that grows with B, q_len or num_shards.  The sizes are only
 * validated: it returns 0 if they are invalid or the device cannot run the
 * kernel.  A library addition with no counterpart in the sources.
 */
uint64_t mla_dcp_decode_partial_workspace_size(int B, int q_len, int num_shards, int has_current);

/*
 * mla_dcp_decode_partial_noalloc -- mla_dcp_decode_partial with no
 * workspace argument and no allocation of any kind.  A library addition
 * with no counterpart in the sources.  It is for callers that cannot hand
 * the library device memory: for example a serving runtime whose memory
 * planner gives all free device memory to its own pool at start-up, so that
 * no buffer can be allocated or lent for a single call.
 *
 * Same arguments, results and errors as mla_dcp_decode_partial (its
 * argument checks run first, in the same order), whose split-shard
 * workspace it takes from a fixed 24 MiB device array inside the library.
 * That holds the workspace of up to 95 CTA pairs with BF16 / FP16 partials,
 * or 47 with FP32 partials.  When this device needs more (FP32 partials on
 * a GPU with more than 47 resident pairs, such as GB300's 76) the call runs
 * as mla_dcp_decode_partial with workspace NULL: every pair takes whole
 * shards and no scratch is used.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) and the kernel's occupancy; make that first call
 *     outside any stream capture.  The address is looked up again if the
 *     device's context changed (after cudaDeviceReset).
 *   - Nothing in the array has to start at zero: every call rewrites each
 *     record it reads.
 *   - All calls on a device share the array: calls that may overlap in time
 *     (on different streams, say) race on it and must be serialised by the
 *     caller.
 */
int mla_dcp_decode_partial_noalloc(const void* q_abs, const void* q_pe, const void* kv_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const void* kv_cur, int B, int q_len, int H, int num_blocks,
                                   int block_size, int max_blocks, int num_shards, float scale,
                                   int in_dtype, int part_dtype, void* o_part, float* lse_part,
                                   int32_t* err_flag, mla_stream_t stream);

/*
 * mla_lse_combine -- merge partials by their log-sum-exps.
 *
 * Defines: [PR] glossary "LSE" and the fourth change (combine without packing the
 * current partial): all history shards plus the local CURRENT partial are merged
 * exactly once; the local partial is read in place (local_output /
 * local_lse) instead of being packed with the others; partials of any of
 * BF16 / FP16 / FP32 are read directly with no FP32 copy ([PR] first change,
 * dtype pass-through).
 *   LSE = ln sum_p exp(lse_p);   o = sum_p exp(lse_p - LSE) * o_p
 * Parts with lse = -inf carry zero weight; if every part is empty, o = 0 and
 * LSE = -inf.  Parts are visited in index order 0..num_parts-1, then local.
 *
 *   o_part    [T, num_parts, H, 512] part_dtype  (T = B * q_len)
 *   lse_part  [T, num_parts, H] float32
 *   o_local   [T, H, 512] part_dtype or NULL;  lse_local [T, H] float32 or NULL
 *             (both NULL or both set)
 *   T >= 1; 1 <= H <= 128; 1 <= num_parts (+1 if local) <= 65
 *   o_latent  [T, H, 512] out_dtype (MLA_BF16 / MLA_FP16 / MLA_FP32)
 *   lse_out   [T, H] float32, or NULL
 */
int mla_lse_combine(const void* o_part, const float* lse_part, int num_parts,
                    const void* o_local, const float* lse_local, int T, int H, int part_dtype,
                    int out_dtype, void* o_latent, float* lse_out, mla_stream_t stream);

/*
 * mla_dcp_combine_exchanged -- the combine on one GPU after the exchange
 * between GPUs.
 *
 * Defines: [PR] the third and fourth changes: after the head-scattered
 * all-to-all each rank combines, for its slice of heads, the HISTORY
 * partials of all ranks plus the CURRENT partial exactly once (the local
 * output / local LSE).  o_recv [num_src][T][parts_per_src][H][512] and
 * lse_recv [num_src][T][parts_per_src][H] are what the all-to-all delivered
 * (block src = the sliced partials of rank src for this rank's heads, H =
 * heads of the slice).  Parts p < hist_parts of every source are history
 * shards; if local_src >= 0, part hist_parts of source local_src (the CURRENT
 * partial, which every rank computes alike) is added once.
 *   LSE = ln sum exp(lse_q);  o = sum exp(lse_q - LSE) o_q  over those parts
 * in the order (src 0, p 0..), (src 1, ...), ..., then the local one; parts
 * with lse = -inf carry no weight.
 *   o_latent [T, H, 512] out_dtype;  lse_out [T, H] float32 or NULL
 *   1 <= num_src * hist_parts (+1 with the local part) <= 96;
 *   1 <= parts_per_src <= 65;  -1 <= local_src < num_src
 */
int mla_dcp_combine_exchanged(const void* o_recv, const float* lse_recv, int num_src,
                              int parts_per_src, int hist_parts, int local_src, int T, int H,
                              int part_dtype, int out_dtype, void* o_latent, float* lse_out,
                              mla_stream_t stream);

/*
 * mla_vup -- batch-major V up-projection.
 *
 * Defines: [PR] code block A (_v_up_proj_batch_major): the latent output is
 * viewed as [T, H, 512], each head is multiplied by W_UV[h] (512 x 128), and
 * the result is returned as [T, H*128] with no transposes in memory.
 *   out[t, h*128 + v] = sum_k o_latent[t, h, k] * W_UV[h, k, v]
 *
 *   o_latent [T, H, 512] dtype;  W_UV [H, 512, 128] dtype
 *   dtype MLA_BF16 or MLA_FP16 (one dtype for both operands; fp32 accumulate)
 *   out      [T, H*128] dtype
 *   1 <= T <= 65536; 1 <= H <= 128;  err_flag as above (may be NULL)
 */
int mla_vup(const void* o_latent, const void* W_UV, int T, int H, int dtype, void* out,
            int32_t* err_flag, mla_stream_t stream);

/*
 * mla_lse_combine_vup -- mla_lse_combine and mla_vup in one launch.  Two
 * exact forms of the same result ([PR] code block A: combine, then the
 * batch-major V-up), chosen per call:
 *   - partials in `dtype` (part_dtype == dtype), at most 64 parts counting
 *     o_local, o_latent NULL: every part's rows are up-projected on the
 *     tensor cores and the LSE-weighted sum is taken in fp32 in the 128-wide
 *     V space (the projection is linear), so the combined latent is never
 *     rounded;
 *   - otherwise: the combined latent of each head is rounded to `dtype` and
 *     fed to the up-projection from on-chip memory.
 * Arguments as in the two calls above; o_latent (written too, if non-NULL)
 * and out use `dtype`.  Parts with lse = -inf are skipped whatever their
 * rows hold.
 *   1 <= T <= 65536
 */
int mla_lse_combine_vup(const void* o_part, const float* lse_part, int num_parts,
                        const void* o_local, const float* lse_local, const void* W_UV, int T,
                        int H, int part_dtype, int dtype, void* out, void* o_latent,
                        float* lse_out, int32_t* err_flag, mla_stream_t stream);

/*
 * mla_gather_kv -- test hook: copy each sequence's paged history into a
 * dense buffer, bit-exactly ([PR] code block B: the HISTORY call reads the
 * cache through block_table / block_size / cp_history_seq_len).
 *   dst[b, t, :] = kv_cache[block_table[b][t / block_size]][t % block_size][:]
 *   for t < seq_lens[b]; rows t >= seq_lens[b] (up to max_len) are zeroed.
 *   elem_bytes 2 (bf16 / fp16); dst [B, max_len, 576] elements.
 *   A block id outside [0, num_blocks) sets MLA_DEV_BAD_BLOCK_ID and its
 *   rows are zeroed.
 */
int mla_gather_kv(const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                  int B, int num_blocks, int block_size, int max_blocks, int max_len,
                  void* dst, int32_t* err_flag, mla_stream_t stream);

/*
 * mla_debug_set_spin_limit -- test hook for the device error path: the
 * number of polls after which a pipeline wait of mla_dcp_decode_partial (and
 * of mla_dcp_decode_partial_noalloc) gives up and records
 * MLA_DEV_WAIT_TIMEOUT; 0 restores the default of 2^22 polls.  It applies
 * to every call launched after it, from any host thread.  With a limit short
 * enough to run out, that call's outputs are unspecified and *err_flag reads
 * MLA_DEV_WAIT_TIMEOUT; the kernel still waits for its own copies and MMAs
 * already issued, frees its tensor memory and returns, so the CUDA context
 * stays usable.  A library addition with no counterpart in the sources.
 */
void mla_debug_set_spin_limit(uint32_t polls);

/* Human-readable text of an mla_status or device error code. */
const char* mla_get_error_string(int status);
const char* mla_device_error_string(int code);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int mla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DCP_H */
