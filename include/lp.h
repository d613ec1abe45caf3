/*
 * lp.h -- C ABI of liblp.so: grammar-constrained logit masking and fused
 * per-row sampling on one GB300 GPU (sm_103a).
 *
 * Operations (each entry point cites the page section that defines it):
 *   lp_apply_token_bitmask   in place, masked logits := -inf
 *   lp_apply_token_bitmask_rows  the same with a per-row flag for the rows to
 *                            mask, and an optional per-row "keeps a token" report
 *   lp_apply_packed_bitmask  out of place, masked logits := fill_value
 *   lp_upload_bitmask        a host-filled bitmask (and row flags) to the device on
 *                            a copy stream, signalled by an event
 *   lp_sample                temperature, top-k ∩ top-p ∩ min-p, Gumbel-max draw
 *   lp_mask_and_sample       the bitmask applied on the fly, then lp_sample
 *   lp_mask_and_sample_slots the same on [slots, rows_per_slot, V] logits with
 *                            per-slot parameters and optional per-row seeds
 *
 * Common conventions
 *   - Logits are a row-major [B, cols] matrix of float32, float16 or bfloat16 with
 *     a row stride in ELEMENTS (stride >= cols).  Only the first vocab_size
 *     columns of a row take part; columns vocab_size..cols-1 are never written.
 *   - The bitmask is a row-major int32 matrix [bitmask_rows, bitmask_words] with a
 *     row stride in WORDS.  Token j of row i is bit (j % 32) of word j / 32, the
 *     word read as an unsigned 32-bit pattern: 1 keeps the token, 0 masks it.
 *     Bits of tokens >= vocab_size are never used.
 *   - vocab_size < 0 selects the default min(cols, bitmask_words * 32).
 *   - indices (optional, int32, device memory): the rows to mask.  The same index
 *     addresses the logits row and the bitmask row.  NULL masks every row
 *     (then bitmask_rows >= B is required).  An index outside
 *     [0, min(B, bitmask_rows)) is skipped on the device: no access, no write.
 *     Indices should be unique; a duplicate gives the same result as one entry.
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller owns every
 *     buffer.  No call allocates memory, and the library keeps no state between
 *     calls beyond one fixed array: the 128 MiB device scratch of
 *     lp_mask_and_sample_noalloc, which the CUDA module reserves (zero-filled) on
 *     every device that loads it, whether or not that entry point is called, and
 *     holds until the process exits.  Calls never synchronise and only enqueue
 *     work on the given stream; a call is safe from several host threads at once
 *     on different buffers.
 *   - Errors: arguments are checked on the host before any launch.  An invalid
 *     argument returns LP_ERR_INVALID_ARGUMENT and launches nothing.  A zero-size
 *     problem returns LP_OK and launches nothing.  A launch failure returns
 *     LP_ERR_CUDA (the CUDA error is left for cudaGetLastError to report).
 */
#ifndef LP_H_
#define LP_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LP_F32 = 0, LP_F16 = 1, LP_BF16 = 2 } lp_dtype;

typedef enum {
  LP_OK = 0,
  LP_ERR_INVALID_ARGUMENT = 1,
  LP_ERR_UNSUPPORTED_DTYPE = 2,
  LP_ERR_CUDA = 3,
  LP_ERR_TOO_LARGE = 4 /* a size past the 32-bit index range of the kernels, or (noalloc)
                          a call needing more scratch than the library's fixed array */
} lp_status;

/*
 * Per-row sampling parameters (Kernel Hub "logits-processor", Ops: every sampling
 * parameter is a scalar broadcast to all rows or a length-B tensor).  The struct
 * itself is HOST memory, read during the call.  Each array pointer is a device
 * pointer to B values, or NULL to use the scalar beside it.
 *   temperature <= 0 (or NaN)  greedy argmax; else logits are divided by it
 *   top_k <= 0                 top-k off; top_k == 1 is greedy
 *   top_p >= 1                 top-p off
 *   min_p <= 0                 min-p off
 *   seed, offset               key of the counter-based draw, with the row index
 */
typedef struct {
  const float* temperature;
  float temperature_scalar;
  const int32_t* top_k;
  int32_t top_k_scalar;
  const float* top_p;
  float top_p_scalar;
  const float* min_p;
  float min_p_scalar;
  uint64_t seed;
  uint64_t offset;
} lp_sampling_params;

/*
 * lp_apply_token_bitmask -- XGrammar "Bitmask Operations",
 * apply_token_bitmask_inplace (the row/token loop; Padding and Indices notes);
 * Kernel Hub "logits-processor", Ops, apply_token_bitmask.
 *
 * For each selected row b and each token j < vocab_size whose bit is 0:
 * logits[b * logits_stride + j] = -inf.  Nothing else changes.
 *   logits         device, [B, cols] with row stride logits_stride (elements)
 *   dt             element type of logits
 *   bitmask        device int32 [bitmask_rows, bitmask_words], stride in words
 * Invalid: B < 0, cols < 0, logits_stride < cols, bitmask_words < 0,
 *   bitmask_stride < bitmask_words, vocab_size > cols,
 *   vocab_size > bitmask_words * 32, num_indices < 0, NULL logits/bitmask with
 *   work to do, num_indices > 0 with NULL indices, bitmask_rows < B without
 *   indices.
 */
lp_status lp_apply_token_bitmask(void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                 int64_t logits_stride, const int32_t* bitmask,
                                 int64_t bitmask_rows, int64_t bitmask_words,
                                 int64_t bitmask_stride, int64_t vocab_size,
                                 const int32_t* indices, int64_t num_indices,
                                 cudaStream_t stream);

/*
 * lp_apply_token_bitmask_rows -- TensorRT-Edge-LLM "Guided Decoder": the mask the
 * apply kernel reads comes with a per-row flag, and a row whose flag is zero is
 * left alone (struct Impl, deviceRowNeedsMask); whether a row's mask admits a
 * token (rowHasAnyToken) is what marks a slot unsatisfiable (fillMasks,
 * unsatisfiableSlots).  Here both run on the device, in the apply's one pass.
 *
 * For each row b with row_needs_mask[b] != 0 (every row when row_needs_mask is
 * NULL) and each token j < vocab_size whose bit is 0:
 * logits[b * logits_stride + j] = -inf.  Nothing else changes.
 *   row_needs_mask  device uint8 [B], or NULL
 *   row_has_token   device int32 [B] written by the call, or NULL: 1 when row b
 *                   keeps at least one token j < vocab_size after the call (an
 *                   unflagged row keeps all of them), else 0; all zeros when
 *                   vocab_size == 0.
 * Other arguments, ownership and errors as lp_apply_token_bitmask without
 * indices: bitmask_rows >= B is required.
 */
lp_status lp_apply_token_bitmask_rows(void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                      int64_t logits_stride, const int32_t* bitmask,
                                      int64_t bitmask_rows, int64_t bitmask_words,
                                      int64_t bitmask_stride, int64_t vocab_size,
                                      const uint8_t* row_needs_mask, int32_t* row_has_token,
                                      cudaStream_t stream);

/*
 * lp_upload_bitmask -- XGrammar "Bitmask Operations", Device: the bitmask is
 * allocated on the CPU and must be copied to the GPU before the apply;
 * TensorRT-Edge-LLM "Guided Decoder", struct Impl: hostBitmask and
 * hostRowNeedsMask stage what the apply kernel reads from deviceBitmask and
 * deviceRowNeedsMask, and captureDraftChains records an event instead of
 * synchronising the stream.
 *
 * Enqueues on copy_stream the copy of rows [0, rows) x words [0, words) of the
 * host bitmask (host_stride words per row) to the device bitmask (device_stride
 * words per row), then, when both are given, of host_flags[0, rows) to
 * device_flags; then records `uploaded` (when not NULL) on copy_stream.  A
 * compute stream that waits on `uploaded` (cudaStreamWaitEvent) sees the new
 * mask, and the copy overlaps whatever else the device runs.  Host buffers must
 * stay untouched until `uploaded` completes, and should be page-locked for the
 * copy to be asynchronous.  No kernel is launched.
 *   device_bitmask  device int32, rows x device_stride words
 *   host_bitmask    host int32, rows x host_stride words
 *   device_flags / host_flags  uint8 [rows], both or neither
 * Invalid: rows < 0, words < 0, a stride < words, only one of the two flag
 * pointers, NULL bitmask pointers with rows > 0 and words > 0.
 */
lp_status lp_upload_bitmask(int32_t* device_bitmask, int64_t device_stride,
                            const int32_t* host_bitmask, int64_t host_stride, int64_t rows,
                            int64_t words, uint8_t* device_flags, const uint8_t* host_flags,
                            cudaStream_t copy_stream, cudaEvent_t uploaded);

/*
 * lp_apply_packed_bitmask -- Modular MAX "apply_packed_bitmask": one fused pass,
 * no boolean tensor; out[b, v] = logits[b, v] where the bit is set, fill_value
 * where it is clear.
 *
 * out receives all B rows x cols columns: the masked result on selected rows for
 * j < vocab_size, a copy of logits everywhere else (unselected rows, columns >=
 * vocab_size).  fill_value is rounded to nearest even into dt.  out may be
 * exactly logits (same pointer and stride: in place); any other overlap is
 * invalid and not detected.  Argument checks as lp_apply_token_bitmask, plus
 * out_stride >= cols and a non-NULL out.
 */
lp_status lp_apply_packed_bitmask(void* out, int64_t out_stride, const void* logits,
                                  lp_dtype dt, int64_t B, int64_t cols,
                                  int64_t logits_stride, const int32_t* bitmask,
                                  int64_t bitmask_rows, int64_t bitmask_words,
                                  int64_t bitmask_stride, float fill_value,
                                  int64_t vocab_size, const int32_t* indices,
                                  int64_t num_indices, cudaStream_t stream);

/*
 * lp_sample -- Kernel Hub "logits-processor", Ops (sample) and How it works.
 *
 * One token id per row of logits[B, vocab_size] (row stride logits_stride):
 *   candidates C = tokens whose logit is above -inf;
 *   C empty -> -1;
 *   greedy (temperature <= 0 or top_k == 1) -> lowest-index argmax of the logits;
 *   else z = logit / temperature, p = softmax(z) over C, keep every v in C with
 *   p_v >= min(max(t_k, t_p, t_m), p_max), where t_k is the k-th largest p,
 *   t_p the p at which the descending cumulative sum first reaches top_p and
 *   t_m = min_p * p_max (a disabled filter contributes 0); the id is
 *   argmax over kept v of z_v + g_v, lowest index on ties, with Gumbel noise
 *   g_v = -log(-log u_v), u_v = ((x >> 9) + 0.5) * 2^-23 and x = word (v & 3) of
 *   Philox4x32-10 (Salmon et al., SC'11) at counter (v >> 2, b, lo32(offset),
 *   hi32(offset)) and key (lo32(seed), hi32(seed)).
 *   out_ids        device int64 [B]
 *   params         host pointer, see lp_sampling_params
 *   workspace      device scratch of at least lp_sample_workspace_bytes(dt, B,
 *                  vocab_size) bytes, 256-byte aligned, owned by the caller.  It
 *                  should be zero-filled before its first use; after that the
 *                  library keeps it valid itself (every call that completes
 *                  leaves the counters in its first 256 + 4 * 16384 bytes zero),
 *                  so one allocation serves any number of calls of the same or
 *                  smaller size.  Results never depend on those counters: after a
 *                  call that failed part-way (LP_ERR_CUDA after the first kernel
 *                  was queued), or on a workspace that was not zero-filled, a
 *                  call still returns correct ids -- a stale row key or pool
 *                  counter only makes rows take the slower re-read path -- and
 *                  resets the counters of the rows it samples.  To restore full
 *                  speed at once, zero those first 256 + 4 * 16384 bytes again
 *                  (or the whole workspace).  Calls that share a workspace must
 *                  be ordered (one stream, or events).  A NULL, misaligned or
 *                  short workspace is LP_ERR_INVALID_ARGUMENT.
 * Each call is two kernels on the stream: a streaming pass over the logits and
 * a per-row finish, the second launched as a programmatic dependent of the
 * first.  An id of -2 means a wait inside the streaming kernel gave up (a copy
 * into shared memory, or the hand-over of a tile's shared state, did not
 * complete within its bounded wait; no such case is known); the call still
 * completes and leaves the workspace valid.
 * Logits are read only.  vocab_size up to 2^31 - 65 and B up to 2^27 are
 * supported; larger sizes return LP_ERR_TOO_LARGE.
 */

/*
 * lp_sample_workspace_bytes -- bytes of device scratch lp_sample and
 * lp_mask_and_sample need for B rows of vocab_size tokens of type dt: per-tile
 * summaries and candidate slots plus a pool for longer candidate buffers --
 * at most about 7% of the logits' size plus 128 MB.  0 for B == 0; -1 for an
 * invalid dt or a negative size.  The result does not depend on the device.
 */
int64_t lp_sample_workspace_bytes(lp_dtype dt, int64_t B, int64_t vocab_size);

lp_status lp_sample(const void* logits, lp_dtype dt, int64_t B, int64_t vocab_size,
                    int64_t logits_stride, const lp_sampling_params* params,
                    int64_t* out_ids, void* workspace, int64_t workspace_bytes,
                    cudaStream_t stream);

/*
 * lp_mask_and_sample -- the bitmask of lp_apply_token_bitmask applied on the fly
 * (masked tokens leave the candidate set; logits are NOT written), then
 * lp_sample.  A masked row whose mask admits no token returns -1
 * (TensorRT-Edge-LLM "Guided Decoder": rowHasAnyToken / unsatisfiableSlots).
 * Rows listed in indices are masked by their own bitmask row, other rows sample
 * unmasked; indices == NULL masks every row.  bitmask == NULL is lp_sample.
 * Argument checks as lp_apply_token_bitmask and lp_sample.
 */
lp_status lp_mask_and_sample(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                             int64_t logits_stride, const int32_t* bitmask,
                             int64_t bitmask_rows, int64_t bitmask_words,
                             int64_t bitmask_stride, int64_t vocab_size,
                             const int32_t* indices, int64_t num_indices,
                             const lp_sampling_params* params, int64_t* out_ids,
                             void* workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * lp_mask_and_sample_slots -- the speculative-verify layout of TensorRT-Edge-LLM
 * "Guided Decoder" (applyMask: logits shaped [activeBatchSize, rowsPerSlot,
 * vocab]; maxRowsPerSlot rows per slot), sampled as Kernel Hub
 * "logits-processor", Ops, sample (per-row parameters; the draw keyed by
 * (seed, row, offset)).
 * lp_mask_and_sample on the B = slots * rows_per_slot rows of a
 * [slots, rows_per_slot, cols] logits tensor (row b = slot * rows_per_slot + r),
 * except that:
 *   - every array in *params holds one value per SLOT (B / rows_per_slot of
 *     them), and a slot's rows take its value;
 *   - seeds, when not NULL, is a device uint64 [B]: row b draws with
 *     (seeds[b], b, offset) instead of (params->seed, b, offset).
 * rows_per_slot = 1 with seeds = NULL is lp_mask_and_sample.
 * Invalid: rows_per_slot < 1, or B not a multiple of rows_per_slot; otherwise
 * as lp_mask_and_sample.
 */
lp_status lp_mask_and_sample_slots(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                   int64_t logits_stride, const int32_t* bitmask,
                                   int64_t bitmask_rows, int64_t bitmask_words,
                                   int64_t bitmask_stride, int64_t vocab_size,
                                   const int32_t* indices, int64_t num_indices,
                                   const lp_sampling_params* params, int64_t rows_per_slot,
                                   const uint64_t* seeds, int64_t* out_ids, void* workspace,
                                   int64_t workspace_bytes, cudaStream_t stream);

/*
 * lp_mask_and_sample_noalloc -- lp_mask_and_sample for callers that cannot
 * allocate device memory themselves: code that must not call cudaMalloc (a
 * caching allocator owns the device, or the call happens where allocation is
 * not allowed, such as inside a captured region) and has no workspace to hand
 * in.  The pages have no counterpart.  Instead of a caller workspace the call
 * uses a 128 MiB device array of the library's own (a file-scope __device__
 * array, zero-filled when the module loads and held by every device that loads
 * the library until the process exits); it allocates nothing.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it; make that
 *     first call before any stream capture.
 *   - Size: the scratch needed, lp_sample_workspace_bytes(dt, B, vocab) for the
 *     vocabulary the call resolves to, must fit in 128 MiB; otherwise the call
 *     returns LP_ERR_TOO_LARGE and launches nothing.  All five benchmark
 *     workloads fit (the largest, 1024 rows of 202048 fp16 tokens, uses about
 *     78 MiB).
 *   - Sharing: every call uses the same array and leaves its counters zero for
 *     the next.  Calls that overlap on the GPU (in flight at once on different
 *     streams, or from several host threads without ordering) race on it and
 *     give undefined ids; order them (one stream, or events).
 * Arguments, results and other errors as lp_mask_and_sample.
 */
lp_status lp_mask_and_sample_noalloc(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                     int64_t logits_stride, const int32_t* bitmask,
                                     int64_t bitmask_rows, int64_t bitmask_words,
                                     int64_t bitmask_stride, int64_t vocab_size,
                                     const int32_t* indices, int64_t num_indices,
                                     const lp_sampling_params* params, int64_t* out_ids,
                                     cudaStream_t stream);

/*
 * lp_philox4x32_10 -- diagnostic: the device's Philox4x32-10 (Salmon et al.,
 * SC'11, 10 rounds) evaluated on n caller-given blocks, so tests can compare the
 * noise stream of lp_sample word for word.
 *   counters  device uint32 [n, 4];  keys  device uint32 [n, 2];
 *   out       device uint32 [n, 4]
 */
lp_status lp_philox4x32_10(const uint32_t* counters, const uint32_t* keys, uint32_t* out,
                           int64_t n, cudaStream_t stream);

/* Static description of a status code; never NULL. */
const char* lp_status_string(lp_status status);

#ifdef __cplusplus
}
#endif

#endif /* LP_H_ */
