/*
 * eb_sampler.h -- C ABI of the B300 (sm_103a) Entropy-Bounded (EB) denoising sampler of
 * DiffusionGemma's block-autoregressive text diffusion.
 *
 * What one sampler step computes (DiffusionGemma model card, "Best practices" section 1,
 * "Diffusion sampling settings"; the Korean model card's "Recommendations" section 1 and
 * the aitrends.kr summary's "Good to know" list say the same):
 *   1. logit shaping: z = x / T with T linear from t_start = 0.8 (step 0) to t_end = 0.4
 *      (step max_steps - 1), max_steps = 48;
 *   2. per canvas position: the full-vocabulary softmax entropy H of z (nats), the
 *      argmax A of the raw logits (first index on ties) and, for still-masked positions,
 *      a Gumbel-max sample Y = argmax_v z_v - ln(-ln u_v) with u_v from Philox4x32-10;
 *   3. adaptive stop (steps >= 1): the mean of H over all L positions is below
 *      stop_entropy = 0.005 AND A equals the previous step's argmax at every position;
 *      then every still-masked position takes A and the canvas is done;
 *   4. otherwise entropy-bounded selection: masked positions sorted by (H, position)
 *      ascending; sorted index i is accepted iff the sum of the entropies before it is
 *      <= entropy_bound = 0.1 (index 0 always); accepted positions commit Y, the rest
 *      stay masked ("fully re-noised");
 *   5. a canvas whose mask empties is complete; at the last step the positions still
 *      masked take A (step cap).
 * The pages give no selection formula; the rule of item 4 is the one this library
 * implements (the longest sorted prefix whose sum minus its maximum stays within the
 * bound).  Items 3 and 5 state the default readings of open points; EB_FLAG_* bits of
 * eb_params.flags select the alternatives (stop statistics over the masked positions only or
 * of the raw logits, sampled-token finalisation).
 *
 * Conventions shared by every entry point:
 *   - every d_* pointer is DEVICE memory owned by the caller; the library allocates
 *     nothing and never synchronises the stream inside eb_sampler_step;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream); all
 *     work is enqueued asynchronously on it;
 *   - argument errors return before any launch and leave every buffer untouched;
 *     eb_last_error() then holds a one-line description (thread-local);
 *   - logits must be finite with |x| < 1e37 (exclude a token with a large negative finite
 *     value such as -1e30); device-detected problems never trap: a canvas whose logits hold
 *     NaN or +-Inf gets EB_STATUS_NONFINITE in its status word and is halted;
 *   - layouts are row-major: logits [B, L, V] with V contiguous; per-position arrays
 *     [B, L]; per-canvas arrays [B];
 *   - tokens use -1 for MASK.
 */
#ifndef EB_SAMPLER_H
#define EB_SAMPLER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EB_OK = 0,
    EB_ERR_INVALID = 1,      /* bad argument; nothing launched */
    EB_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed */
    EB_ERR_UNSUPPORTED = 3,  /* valid but unsupported shape / device */
    EB_ERR_WORKSPACE = 4,    /* workspace missing or smaller than eb_workspace_bytes() */
    EB_ERR_CALLBACK = 5      /* the logits callback of eb_sample_canvas returned non-zero */
} eb_status;

/* Logit element types: binary32, bfloat16, and OCP FP8 e4m3 (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN) for the streaming entry points. */
typedef enum { EB_F32 = 0, EB_BF16 = 1, EB_FP8_E4M3 = 2 } eb_dtype;

/* Canvas status word d_status[b]: the low byte is the stop reason. */
#define EB_RUNNING 0
#define EB_STOP_ADAPTIVE 1       /* mean entropy < stop_entropy and argmax stable */
#define EB_STOP_COMPLETE 2       /* every position committed by selection */
#define EB_STOP_CAP 3            /* the last step (max_steps - 1) was reached */
#define EB_STATUS_NONFINITE 0x100 /* or-ed in: NaN / +-Inf logits seen; canvas halted */
#define EB_STATUS_TIMEOUT 0x200   /* or-ed in: a bounded device wait gave up; canvas halted */
#define EB_SLOT_IDLE 0x400        /* eb_sample_blocks: a slot holding no block */
#define EB_STATUS_CHECK 0x800     /* or-ed in (checked build only): a device bounds check failed
                                     (eb_check_word); canvas halted */

typedef struct {
    int32_t max_steps;     /* 48 */
    float t_start;         /* 0.8: temperature at step 0 */
    float t_end;           /* 0.4: temperature at step max_steps - 1 */
    float entropy_bound;   /* 0.1 */
    float stop_entropy;    /* 0.005 (strict <) */
    uint32_t flags;        /* 0 or EB_FLAG_* bits below; other bits are refused */
    uint64_t seed;         /* Philox key (low, high 32 bits) of the Gumbel noise */
} eb_params;

/* Reading variants (bits of eb_params.flags).  The model card leaves two points of the stop
 * rule open; the default reading (flags 0) is: the mean entropy and the argmax-stability test
 * run over all L positions, committed ones included ("mean model entropy over the whole
 * canvas", DiffusionGemma model card, Best practices section 1, adaptive stop), and positions
 * still masked at an adaptive stop or at the step cap take the current argmax.
 *   EB_FLAG_STOP_MASKED_ONLY: the stop statistics run over the positions still masked at the
 *     start of the step (mean_entropy then reports that mean);
 *   EB_FLAG_FINALIZE_SAMPLED: positions finalised at an adaptive stop or at the step cap take
 *     their sampled token instead of the argmax;
 *   EB_FLAG_STOP_RAW_ENTROPY: the stop rule's mean uses the entropy of the raw logits (T = 1)
 *     instead of the shaped ones (selection still uses the shaped entropy; mean_entropy then
 *     reports the raw mean).  It costs a second, sampling-free pass over the logits; the fused
 *     entry point refuses it (EB_ERR_UNSUPPORTED), as its logits are never stored. */
#define EB_FLAG_STOP_MASKED_ONLY 2u
#define EB_FLAG_FINALIZE_SAMPLED 4u
#define EB_FLAG_STOP_RAW_ENTROPY 8u

/* Diagnostic bit of eb_params.flags.  The fused unembedding kernel of eb_unembed_sample then
 * withholds its first operand load and lets each device wait poll only a few thousand times.
 * Its bounded waits therefore give up: the kernel waits for the copies it did issue, frees its
 * tensor memory and returns, and every running canvas of the call ends with EB_STATUS_TIMEOUT
 * (and EB_STATUS_NONFINITE, as its statistics are empty) while the CUDA context stays usable.
 * It exists to exercise that failure path without a fault; the other entry points ignore it.
 * The model card has no counterpart. */
#define EB_FLAG_DIAG_STALL 1u

/* Fills *p with the model card's recommended settings (48, 0.8, 0.4, 0.1, 0.005) and
 * seed 0.  Returns EB_ERR_INVALID on NULL. */
eb_status eb_default_params(eb_params *p);

/* Temperature of `step` on the linear schedule: t_start + (t_end - t_start) * step /
 * (max_steps - 1), t_start when max_steps == 1.  Evaluated in binary32. */
float eb_temperature(const eb_params *p, int step);

/* Bytes of device workspace eb_sampler_step / eb_sample_canvas need for B canvases of L
 * positions (V and dtype do not change it today but are part of the contract).  The
 * workspace must be 256-byte aligned; its contents need no initialisation. */
size_t eb_workspace_bytes(int B, int L, int V, eb_dtype dtype);

/*
 * One EB sampler step over B canvases (items 1-5 above).
 *
 *   params         sampler settings (host pointer, read during the call only)
 *   B, L, V        canvases, positions per canvas (1..1024), vocabulary (1..2^31-1)
 *   dtype          element type of d_logits (EB_F32, EB_BF16 or EB_FP8_E4M3)
 *   d_logits       [B, L, V] logits of this step (read only)
 *   step           denoising step index s (0-based, < params->max_steps); keys the
 *                  Gumbel noise and the stop / cap rules
 *   temperature    > 0: use this T; <= 0: use eb_temperature(params, step)
 *   d_mask         [B, L] u8 in/out, 1 = masked
 *   d_tokens       [B, L] i32 in/out, committed token or -1
 *   d_prev_argmax  [B, L] i32 in/out, argmax of the previous step (-1 before step 0)
 *   d_status       [B] i32 in/out; canvases whose status is not EB_RUNNING are skipped
 *   d_steps_taken  [B] i32 out (written when a canvas stops: step + 1); may be NULL
 *   d_entropy      [B, L] f32 out: H in nats (running canvases only)
 *   d_argmax       [B, L] i32 out: A
 *   d_sampled      [B, L] i32 out: Y for masked positions, -1 otherwise
 *   d_selected     [B, L] u8 out: 1 where a token was committed at this step
 *   d_committed    [B] i32 out: positions committed at this step; may be NULL
 *   d_mean_entropy [B] f32 out: mean H of the canvas; may be NULL
 *   d_workspace    eb_workspace_bytes(B, L, V, dtype) bytes, 256-byte aligned
 *   stream         cudaStream_t
 * B == 0 is a no-op.  Returns EB_OK once the work is enqueued.
 */
eb_status eb_sampler_step(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                          const void *d_logits, int step, float temperature,
                          uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                          int32_t *d_status, int32_t *d_steps_taken,
                          float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                          uint8_t *d_selected, int32_t *d_committed, float *d_mean_entropy,
                          void *d_workspace, size_t workspace_bytes, void *stream);

/*
 * eb_sampler_step without a workspace argument.  There is no counterpart in the pages: this
 * entry point exists for callers that cannot call cudaMalloc.  For example:
 *   - a host process whose device memory is all reserved up front by its own pool, so that a
 *     further allocation would fail;
 *   - a plugin that runs inside someone else's runtime, where only that runtime may allocate;
 *   - a latency-critical loop where the implicit synchronisation of an allocation is not
 *     acceptable.
 * The per-row partial states live instead in one fixed array of device memory inside this
 * library, sized for at most EB_NOALLOC_MAX_ROWS canvas positions (B * L).  That is
 * 1,245,696 bytes, and every device that loads the library holds them until the process exits.
 *
 * Arguments, results and errors are those of eb_sampler_step, with the workspace supplied by
 * the library.  B * L above EB_NOALLOC_MAX_ROWS returns EB_ERR_UNSUPPORTED and launches
 * nothing.  The call allocates no memory, neither itself nor through a library.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current, and caches it for the life of the process.  Make that first call before
 * any stream capture.  A cudaDeviceReset (or any other teardown of the device's primary
 * context) voids the cached address; this entry point is not supported after one.
 *
 * All calls share the one array, and it keeps whatever the last call left in it.  Nothing in
 * it needs to start at zero: each call overwrites what it reads later.  Two calls whose work
 * overlaps on the GPU (different streams, or different host threads without ordering) race on
 * the array and may return wrong results.  Order them on one stream, or use eb_sampler_step
 * with separate workspaces.
 */
#define EB_NOALLOC_MAX_ROWS 8192

eb_status eb_sampler_step_noalloc(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                                  const void *d_logits, int step, float temperature,
                                  uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                                  int32_t *d_status, int32_t *d_steps_taken,
                                  float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                                  uint8_t *d_selected, int32_t *d_committed, float *d_mean_entropy,
                                  void *stream);

/* Logits provider of the denoising loop: enqueue, on `stream`, the logits of `step`
 * into d_logits [B, L, V] (the denoiser).  It may read d_tokens / d_status (device) to
 * condition on the canvas and to skip halted canvases.  Returns 0 on success. */
typedef int (*eb_logits_fn)(void *user, int step, const int32_t *d_tokens,
                            const int32_t *d_status, void *d_logits, void *stream);

/*
 * The denoising loop over B independent canvases: for s = start_step .. max_steps-1,
 * logits_fn(s) then eb_sampler_step(s) with the schedule temperature.  Each canvas
 * stops on its own (its later steps cost no sampler work); the loop ends early when
 * every canvas has stopped, checked on the host every `poll_every` steps (0 = never:
 * run to max_steps; a check copies the B status words back and waits for the stream).  Resuming at
 * start_step with the state of an earlier call reproduces an uninterrupted run.
 *
 *   d_logits            [B, L, V] buffer the callback fills each step
 *   d_mask .. d_steps_taken   canvas state as in eb_sampler_step (in/out)
 *   d_committed_per_step [B, max_steps] i32 out or NULL: positions committed at step s
 *   d_mean_entropy_per_step [B, max_steps] f32 out or NULL: mean H at step s
 *   d_entropy, d_argmax, d_sampled, d_selected: as in eb_sampler_step, holding the last
 *                        step's values
 *   steps_run            host out (may be NULL): sampler steps enqueued
 * Returns EB_ERR_CALLBACK (after enqueuing nothing further) if logits_fn fails.
 */
eb_status eb_sample_canvas(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                           eb_logits_fn logits_fn, void *user, void *d_logits, int start_step,
                           uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                           int32_t *d_status, int32_t *d_steps_taken,
                           int32_t *d_committed_per_step, float *d_mean_entropy_per_step,
                           float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                           uint8_t *d_selected, void *d_workspace, size_t workspace_bytes,
                           int poll_every, int *steps_run, void *stream);

/* Denoiser of the block driver: enqueue, on `stream`, the logits of every occupied slot b
 * (d_slot_block[b] >= 0: the block it holds) at that block's own step d_slot_step[b] into
 * d_logits [B, L, V]; slots with d_slot_block[b] < 0 are idle and may be left as they are.
 * d_tokens [B, L] holds each slot's canvas (committed tokens, -1 where masked).  All four
 * arrays are device memory.  Returns 0 on success. */
typedef int (*eb_block_logits_fn)(void *user, int B, const int32_t *d_slot_block,
                                  const int32_t *d_slot_step, const int32_t *d_tokens,
                                  void *d_logits, void *stream);

/* Bytes of device workspace eb_sample_blocks needs for B slots of L positions: the step
 * workspace plus the slots' canvas state.  256-byte aligned; no initialisation needed. */
size_t eb_blocks_workspace_bytes(int B, int L, int V, eb_dtype dtype);

/*
 * Block driver with continuous batching.  DiffusionGemma generates block-autoregressively:
 * a canvas is denoised until done, then the model moves on to the next canvas (model card,
 * "Model overview", multi-canvas sampling), and each canvas stops on its own step count
 * ("Best practices" section 1, adaptive stop).  The pages give no serving loop; this is the
 * plainest one that keeps every slot busy.  n_blocks canvases
 * ("blocks") of L positions are generated on B slots.  Block k starts all masked at step 0,
 * with k as its canvas id in the Gumbel noise's Philox counter (so its result does not depend
 * on the slot it runs in), and follows the denoising loop of eb_sample_canvas: each
 * iteration, logits_fn fills the occupied slots' logits, one sampler step runs with every
 * slot at its block's own step and schedule temperature, and a slot whose block stopped
 * writes the block's tokens, step count and stop reason and takes the next block, or goes
 * idle (EB_SLOT_IDLE) when none is left.  Blocks are handed to slots in the order the slots
 * free up, which the results do not depend on.
 *
 *   params            as in eb_sampler_step (flags included)
 *   B                 slots (>= 1); L, V, dtype as in eb_sampler_step
 *   logits_fn, user   the denoiser (above); d_logits its [B, L, V] output buffer
 *   n_blocks          blocks to generate (0 .. 2^24)
 *   d_block_tokens    [n_blocks, L] i32 out: each block's final tokens
 *   d_block_steps     [n_blocks] i32 out or NULL: steps the block ran
 *   d_block_status    [n_blocks] i32 out or NULL: its stop reason (EB_STOP_* plus status bits)
 *   d_workspace       eb_blocks_workspace_bytes(B, L, V, dtype) bytes, 256-byte aligned
 *   poll_every        read the finished-block count back every `poll_every` iterations and
 *                     stop once all are done (0: run the bound of n_blocks * max_steps
 *                     iterations, the idle ones costing no sampler work)
 *   iterations_run    host out (may be NULL): iterations enqueued
 * Returns EB_ERR_CALLBACK (after enqueuing nothing further) if logits_fn fails.
 */
eb_status eb_sample_blocks(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                           eb_block_logits_fn logits_fn, void *user, void *d_logits, int n_blocks,
                           int32_t *d_block_tokens, int32_t *d_block_steps, int32_t *d_block_status,
                           void *d_workspace, size_t workspace_bytes, int poll_every,
                           int *iterations_run, void *stream);

/*
 * Fused unembedding + sampler step.  The logits of the step are the product of the decoder's
 * final hidden states and the unembedding matrix, logits = h W (the model card's decoder
 * emits full-vocabulary logits for every canvas position at every step, "Best practices"
 * section 1 consumes them); this entry point computes that product on the tensor cores and
 * feeds every accumulator tile straight into the row statistics of item 2, so the [B*L, V]
 * logits are never written to memory.  Items 1-5 then run exactly as in eb_sampler_step, on
 * the fp32 accumulator values as the raw logits.
 *
 *   B, L           canvases and positions per canvas; M = B * L rows of h
 *   K              hidden width (a positive multiple of 8)
 *   V              vocabulary (a positive multiple of 8)
 *   d_h            [M, K] bf16, row-major (K contiguous), 16-byte aligned (read only)
 *   d_W            [K, V] bf16, row-major (V contiguous), 16-byte aligned (read only)
 *   the other arguments as in eb_sampler_step; the workspace must hold
 *   eb_unembed_workspace_bytes(B, L, K, V) bytes, 256-byte aligned.
 * Needs a device with tcgen05 tensor cores (sm_10x); EB_ERR_UNSUPPORTED otherwise.
 */
size_t eb_unembed_workspace_bytes(int B, int L, int K, int V);

eb_status eb_unembed_sample(const eb_params *params, int B, int L, int K, int V, const void *d_h,
                            const void *d_W, int step, float temperature, uint8_t *d_mask,
                            int32_t *d_tokens, int32_t *d_prev_argmax, int32_t *d_status,
                            int32_t *d_steps_taken, float *d_entropy, int32_t *d_argmax,
                            int32_t *d_sampled, uint8_t *d_selected, int32_t *d_committed,
                            float *d_mean_entropy, void *d_workspace, size_t workspace_bytes,
                            void *stream);

/* The same tensor-core product written out: d_logits [M, V] fp32 (row-major) = h W with h
 * [M, K] and W [K, V] bf16 as above.  For callers that need the logits themselves. */
eb_status eb_unembed_logits(int M, int K, int V, const void *d_h, const void *d_W, float *d_logits,
                            void *stream);

/* Instrumentation: CUDA events (cudaEvent_t as void*) to record on the stream right
 * before and right after the row-statistics kernel (the streaming one, or the fused
 * unembedding one) of the NEXT eb_sampler_step / eb_sample_canvas step / eb_unembed_sample /
 * eb_unembed_logits call enqueued by the calling thread (one-shot; NULL, NULL clears).
 * Lets a caller time the dominant kernel alone with CUDA events. */
eb_status eb_set_profile_events(void *k1_begin, void *k1_end);

/* Short English name of a status code (static storage). */
const char *eb_status_string(eb_status s);

/* Description of the last error returned on the calling thread ("" if none). */
const char *eb_last_error(void);

/* The checked debug build.  The same sources compiled with -DEB_CHECKS (the library
 * libeb_sampler_checks.so next to libeb_sampler.so) test, before every access whose index the
 * streaming and selection kernels compute (partial-state slots, row segments, partition units,
 * selected positions), that it lies inside its array.  A failed check skips the access, sets a
 * bit in a device word of the library (1: partial-state slot, 2: row or position, 4: row
 * segment, 8: partition units) and never traps; the selection kernel then or-s
 * EB_STATUS_CHECK into the status of the canvases it decides, which halts them.  The word
 * stays set until read with clear = 1.  The checks cover the streaming path; the fused
 * kernel's own writes are not checked.
 *
 * eb_checks_enabled: 1 in the checked build, 0 in the normal one.
 * eb_check_word: the device word's bits (0 in the normal build); clear != 0 resets it to 0.
 * Synchronous (it copies the word to the host); returns 0 if the copy fails. */
int eb_checks_enabled(void);
uint32_t eb_check_word(int clear);

#ifdef __cplusplus
}
#endif

#endif /* EB_SAMPLER_H */
