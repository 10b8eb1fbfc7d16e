/*
 * eb_synth.h -- C ABI of the seeded synthetic-input generator used by the tests and the
 * benchmark as a stand-in denoiser.  It holds none of the sampler's arithmetic.
 *
 * Logits [B, L, V] (row-major, V contiguous) are a Gaussian background plus one planted
 * peak per canvas position:
 *   x[b, p, v] = sigma * n[b, p, v] + (v == t_p ? h_p(s) : 0),
 *   h_p(s) = ((base_scale * u_p) + base_lo) + growth[b] * s,
 * with n from Box-Muller on Philox4x32-10 words (key = seed[b], counter = (v / 4, p, s,
 * 2 << 24 | b)), and t_p = (w0 * V) >> 32, u_p = ((w1 >> 9) + 1/2) 2^-23 from the words of
 * counter (0, p, 0, 3 << 24 | b).  Every binary32 operation is rounded to nearest even in a
 * fixed order (no fused multiply-add), so the values are bit-identical to the numpy
 * generator of the eb_synth Python package; bfloat16 rounds to nearest even, e4m3 to nearest
 * even with saturation at 448.
 *
 * Pointers prefixed d_ are device memory owned by the caller; `stream` is a cudaStream_t
 * passed as void*.  Functions return 0 on success, non-zero on a bad argument or a CUDA
 * launch error (nothing is enqueued on a bad argument).
 */
#ifndef EB_SYNTH_H
#define EB_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EB_SYNTH_MAX_B 64

typedef struct {
    int32_t B, L, V;
    int32_t dtype;                       /* 0 = binary32, 1 = bfloat16, 2 = FP8 e4m3 */
    float sigma, base_lo, base_scale;
    float growth[EB_SYNTH_MAX_B];        /* per canvas */
    uint64_t seed[EB_SYNTH_MAX_B];       /* per canvas */
} eb_synth_recipe;

/* Writes the logits of `step` into d_logits [B, L, V].  Canvases b with d_status != NULL
 * and d_status[b] != 0 are skipped (their rows are left as they are). */
int eb_synth_logits(const eb_synth_recipe *recipe, int step, const int32_t *d_status,
                    void *d_logits, void *stream);

/* Same signature as eb_logits_fn of eb_sampler.h: user = const eb_synth_recipe* (host). */
int eb_synth_logits_callback(void *user, int step, const int32_t *d_tokens,
                             const int32_t *d_status, void *d_logits, void *stream);

/* Denoiser of the block driver: slot b of d_logits [B_slots, L, V] receives the logits of
 * recipe canvas k = d_slot_block[b] (0 <= k < recipe->B; other slots are left as they are) at
 * step d_slot_step[b], exactly as eb_synth_logits writes canvas k at that step. */
int eb_synth_slot_logits(const eb_synth_recipe *recipe, int B_slots, const int32_t *d_slot_block,
                         const int32_t *d_slot_step, void *d_logits, void *stream);

/* Same signature as eb_block_logits_fn of eb_sampler.h: user = const eb_synth_recipe* (host). */
int eb_synth_block_callback(void *user, int B, const int32_t *d_slot_block, const int32_t *d_slot_step,
                            const int32_t *d_tokens, void *d_logits, void *stream);

/* Fused-unembedding inputs: h [M, K] = N(0,1) and W [K, V] = sigma_w * N(0,1) plus `bias`
 * at column c_k = (w0 * V) >> 32 of each row k (counter (0, k, 0, 6 << 24)), as bfloat16.
 * h uses counter (j / 4, m, 0, 5 << 24) over its K columns j; W uses (v / 4, k, 0, 7 << 24). */
int eb_synth_unembed_inputs(uint64_t seed, int M, int K, int V, float sigma_w, float bias,
                            uint16_t *d_h, uint16_t *d_W, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EB_SYNTH_H */
