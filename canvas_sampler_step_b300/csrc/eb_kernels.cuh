// eb_kernels.cuh -- device code of the B300 (sm_103a) Entropy-Bounded (EB) denoising sampler
// step of DiffusionGemma (model card, "Best practices" section 1, "Diffusion sampling
// settings": at most 48 steps, temperature 0.8 -> 0.4 for logit shaping, lowest-entropy
// selection under the entropy bound 0.1, full re-noising of the unselected tokens, adaptive
// stop at mean entropy < 0.005 with an argmax stable over two consecutive steps).
//
// k1_rowstats (one launch per step) streams the [B, L, V] logits exactly once.
//   * Work split.  Row r of a running canvas weighs nvec * w (w = w_masked for masked rows,
//     which also draw Gumbel noise, w_unmasked otherwise; rows of halted canvases weigh 0).
//     The prefix sums P of the weights are cut into G equal ranges, one per warp (16 warps per
//     CTA, one CTA per SM), so warps finish together even though masked rows cost more
//     instructions per byte, and halted canvases cost nothing.  Unit u runs on CTA u mod G/16,
//     so every SM mixes masked and unmasked work.  Unit g writes one partial state for every
//     row its range touches to slot (row + g) of the workspace (the (row, unit) pairs form a
//     staircase, so row + g is unique).
//   * Data movement.  Each lane copies the 16-byte vectors it will consume (two per batch;
//     one for e4m3, whose vector holds 16 logits) with cp.async (L2 evict-first, no L1) into
//     its own shared-memory slots four batches ahead of use, and waits only for its own
//     oldest group; the slot offset and the global pointer advance by constants.  Whole
//     batches run without bounds checks; the ragged last batch is staged in the same ring
//     (vectors past the segment zero-filled without a read) and taken vector by vector.  (A TMA
//     bulk-copy ring with a producer warp measured slower on this workload, its consumers
//     idling on the ring's barriers; register double buffering had too little in flight.)
//   * Per element: t = x * log2(e)/T - xm * log2(e)/T, e = 2^t (MUFU), S += e, T2 += t e,
//     with xm the warp's running maximum of the raw logits (first index kept for the argmax);
//     the FMAs and adds run on packed f32x2 pairs.  H = ln 2 (log2 S - T2 / S) after merging.
//     A batch takes one new-maximum vote, so the rare rescale stays a branch.
//   * Gumbel-max for masked rows: with u from a Philox4x32-10 word and E = -ln u, the sample
//     maximises z - ln E.  Since E >= 1 - u, an entry can beat the best score so far only if
//     1 - u < 2^t K, K = 2^(xm log2e / T - best log2e); one candidate vote per batch.  A
//     segment's first batch sets the threshold from the score estimates of all its entries
//     (their maximum less the estimate's error).  Entries that pass later (about one per
//     record of the best score) take the exact score z - logf(-log1pf(-(1 - u))) in an
//     out-of-line function, handed the Philox words already drawn; the warp shares its best
//     score when it moves.
//   * Optional per-canvas step, temperature and Philox canvas id (the block driver), and a
//     sampling-free raw mode at T = 1 (the raw-logit entropy of the stop rule's variant).
// k2_select (one CTA per canvas) copies the canvas's contiguous range of partial states to
// shared memory, merges each row's partials in ascending unit order (deterministic), runs the
// stop test, the entropy-bounded selection and the commit / re-mask / finalisation.  Sums of
// entropies are exact 64-bit fixed point (2^-40 nats).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "eb_sampler.h"

namespace ebk {

// ---------------------------------------------------------------- launch geometry
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kMaxWeightedRows = 4096;
constexpr int kK2Threads = 512;                     // two threads per canvas row
constexpr int kMaxL = 1024;
constexpr int kMaxGrid = 8192;
constexpr int kWeightUnmasked = 11;                // relative cost of a vector of an unmasked row
constexpr int kWeightMasked = 33;                  // ... and of a masked row (3 : 1, tuned on the mixed step)
constexpr uint32_t kWaitLimit = 1u << 26;           // mbarrier polls before giving up
constexpr uint32_t kDiagWaitLimit = 1u << 12;       // ... under the diagnostic stall flag

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kEmptyMax = -1.0e30f;               // running max of a slice that saw nothing
constexpr float kCandSlack = 1.0f + 1.0f / 256.0f;  // relative slack of the candidate test
constexpr float kCandAdd = 1.00000011920928955f;    // 1 + 2^-23: additive slack over 1 - 2^-24
constexpr float kOneMinusHalfUlp = 0.99999994039535522f;  // 1 - 2^-24
constexpr uint32_t kStreamGumbel = 1u;

constexpr int kPartialTimeout = 1;                  // Partial::flags: a wait gave up
constexpr int kPartialNonfinite = 2;                // Partial::flags: NaN reached the sums

// Philox4x32-10 round keys (k0 + r 0x9E3779B9, k1 + r 0xBB67AE85), r = 0..9, precomputed
// on the host; as a kernel parameter every key xor reads the constant bank.
struct RoundKeys {
    uint32_t k[20];
};

// Per-(row, CTA) partial state.  xm: max raw logit of the slice (kEmptyMax if empty);
// S, T2: sums of 2^t and t 2^t with t = (x - xm) c, c = log2(e)/T; ai: first index of xm;
// best / bi: best Gumbel score z - ln E and its index (-inf / -1 if none).
struct __align__(16) Partial {
    float xm, S, T2;
    int ai;
    float best;
    int bi;
    int flags;
    int pad;
};

struct RowState {
    float xm, S, T2;
    int ai;
    float best;
    int bi;
};

// Bounds checks of the debug build (compiled with -DEB_CHECKS): a failed check records a bit
// in a device word and the access it guards is skipped; nothing traps.  The selection kernel
// then or-s EB_STATUS_CHECK into the status of the canvases it decides.  In the normal build
// EB_CHECK(c) is the constant true and costs nothing.
#ifdef EB_CHECKS
__device__ unsigned int g_check_word;
__device__ __forceinline__ bool eb_check_ok(bool ok, unsigned int bit)
{
    if (!ok) atomicOr(&g_check_word, bit);
    return ok;
}
#define EB_CHECK(cond, bit) ::ebk::eb_check_ok((cond), (bit))
#else
#define EB_CHECK(cond, bit) true
#endif
constexpr unsigned int kCheckPartialSlot = 1u;   // a partial-state slot outside the workspace
constexpr unsigned int kCheckRow = 2u;           // a row or position index outside its array
constexpr unsigned int kCheckSegment = 4u;       // a row segment outside its row
constexpr unsigned int kCheckUnits = 8u;         // a row's partition units out of order or range

struct K1Args {
    const void *logits;
    const uint8_t *mask;
    const int32_t *status;
    Partial *partials;
    uint32_t *prefix_out;   // [rows + 1] weight prefix (weighted mode; written by CTA 0)
    int2 *rowunits;         // [rows]: first and last partition unit of each row (written here)
    long long nvec_row;     // 16-byte vectors per row (elements per row on the scalar path)
    long long row_bytes;
    int rows;
    int L;
    int G;
    int step;
    int weighted;           // 1: masked-weighted prefix partition, 0: uniform closed form
    float c;                // log2(e) / T
    float invT;             // 1 / T
    RoundKeys keys;
    // per-canvas overrides of step, c and 1/T and the canvas id of the Philox counter, or null
    // (continuous batching: every slot's canvas is at its own step)
    const int32_t *canvas_step;
    const int32_t *canvas_id;
    const float *canvas_c;
    const float *canvas_invT;
    int raw;                // 1: every row as unmasked (no sampling), for the raw-logit entropy
#ifdef EB_CHECKS
    long long nslots;       // partial-state slots in the workspace (bounds checks)
#endif
};

struct K2Args {
    const Partial *partials;
    const uint32_t *prefix;  // weighted mode: [rows + 1]
    const int2 *rowunits;    // [rows]: first and last partition unit of each row
    uint8_t *mask;
    int32_t *tokens;
    int32_t *prev_argmax;
    int32_t *status;
    int32_t *steps_taken;
    float *entropy;
    int32_t *argmax;
    int32_t *sampled;
    uint8_t *selected;
    int32_t *committed;        // [B] or null
    float *mean_entropy;       // [B] or null
    int32_t *committed_hist;   // [B, max_steps] or null
    float *mean_hist;          // [B, max_steps] or null
    long long nvec_row;
    int rows;
    int L;
    int G;
    int step;
    int max_steps;
    int weighted;
    float c;
    long long bound_q;         // entropy_bound in 2^-40 nats (rounded down)
    long long stop_q;          // stop_entropy * L in 2^-40 nats (rounded up): mean < stop
    double stop_entropy;       // for the masked-only statistics (threshold per masked count)
    const int32_t *canvas_step;  // per-canvas step, or null (then `step`)
    const float *canvas_c;       // per-canvas c, or null (then `c`)
    int stop_masked_only;      // EB_FLAG_STOP_MASKED_ONLY
    int finalize_sampled;      // EB_FLAG_FINALIZE_SAMPLED
    // EB_FLAG_STOP_RAW_ENTROPY: partial states of a second pass over the same logits at T = 1
    // (all rows unmasked, its own partition); the stop statistic then sums their entropies
    const Partial *raw_partials;
    const uint32_t *raw_prefix;
    const int2 *raw_rowunits;
    int raw_G, raw_weighted;
    int k3_g;                  // > 0: partials come from the fused unembedding kernel, whose
                               // row block mb, group rank j < k3_g and column group hh <
                               // k3_groups write slot ((mb k3_g + j) k3_groups + hh) 128 + row % 128
    int k3_groups;
#ifdef EB_CHECKS
    long long nslots;          // partial-state slots in the workspace (bounds checks)
#endif
};

// ---------------------------------------------------------------- small device helpers

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed pairs of binary32 values in one 64-bit register (Blackwell f32x2 arithmetic: one
// instruction per two lanes' worth of FADD / FFMA / FMUL).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void upk2(f32x2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Philox4x32-10 (Salmon et al., SC'11): per round two 32x32->64 products of counter words 0
// and 2, high halves xored with the other counter words and the round key.
__device__ __forceinline__ uint4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                        const RoundKeys &K)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ K.k[2 * r];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ K.k[2 * r + 1];
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Row constants of Philox4x32-10 along one canvas row.  Counter words 1-3 (position p, step
// s, stream and canvas sw) are the same for every block of a row, so round 0's product of word
// 2, round 0's new word 0 and round 1's product of that word depend on the row alone; the
// xor partners below fold them with the round keys.
struct PhiloxRow {
    uint32_t c1x;   // round 0: sw ^ k0'   (partner of hi(M0 c0))
    uint32_t c2x;   // round 1: lo(M1 s) ^ k1  (partner of hi(M1 c2))
    uint32_t c3x;   // round 1: hi(M0 n0) ^ k1' (partner of c3)
    uint32_t c5x;   // round 2: lo(M0 n0) ^ k2' (partner of hi(M0 c0))
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t p, uint32_t s, uint32_t sw, const RoundKeys &K)
{
    const uint64_t ps = (uint64_t)0xCD9E8D57u * s;
    const uint32_t n0 = (uint32_t)(ps >> 32) ^ p ^ K.k[0];      // round 0's new word 0
    const uint64_t pn = (uint64_t)0xD2511F53u * n0;               // round 1's first product
    PhiloxRow r;
    r.c1x = sw ^ K.k[1];
    r.c2x = (uint32_t)ps ^ K.k[2];
    r.c3x = (uint32_t)(pn >> 32) ^ K.k[3];
    r.c5x = (uint32_t)pn ^ K.k[5];
    return r;
}

// Philox4x32-10 of counter (c0, p, s, sw) from the row constants of (p, s, sw): the same
// words as philox(c0, p, s, sw, K), with the row-constant work of rounds 0-2 left out.
__device__ __forceinline__ uint4 philox_row_block(uint32_t c0, const PhiloxRow &R, const RoundKeys &K)
{
    const uint64_t a = (uint64_t)0xD2511F53u * c0;                // round 0
    const uint32_t x2 = (uint32_t)(a >> 32) ^ R.c1x;
    const uint32_t x3 = (uint32_t)a;
    const uint64_t b = (uint64_t)0xCD9E8D57u * x2;                // round 1
    uint32_t w0 = (uint32_t)(b >> 32) ^ R.c2x;
    uint32_t w1 = (uint32_t)b;
    uint32_t w2 = x3 ^ R.c3x;
    uint32_t w3;
    {                                                              // round 2
        const uint64_t p0 = (uint64_t)0xD2511F53u * w0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * w2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ w1 ^ K.k[4];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ R.c5x;
        w1 = (uint32_t)p1;
        w3 = (uint32_t)p0;
        w0 = n0;
        w2 = n2;
    }
#pragma unroll
    for (int r = 3; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * w0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * w2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ w1 ^ K.k[2 * r];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ w3 ^ K.k[2 * r + 1];
        w1 = (uint32_t)p1;
        w3 = (uint32_t)p0;
        w0 = n0;
        w2 = n2;
    }
    return make_uint4(w0, w1, w2, w3);
}

// f = 1 + (0x7FFFFF - j) 2^-23 for j = low 23 bits of w, so that 1 - u = f - (1 - 2^-24)
// exactly, u = (j + 1/2) 2^-23 being the entry's uniform.
__device__ __forceinline__ float one_minus_u_plus(uint32_t w)
{
    return __uint_as_float((w & 0x7FFFFFu) ^ 0x3FFFFFFFu);
}

// u' = 1 + j 2^-23 for j = low 23 bits of w: then 1 - u = 2 - u' - 2^-24 exactly.  An entry can
// beat the best score only if 1 - u < e K (e = 2^t, K = cand_scale), i.e. u' + e K > 2 - 2^-24; a
// single rounding of u' + e K then gives a value >= 2, which sets bit 30 of its binary32 bits.
__device__ __forceinline__ float u_prime(uint32_t w)
{
    return __uint_as_float((w & 0x7FFFFFu) | 0x3F800000u);
}

constexpr uint32_t kCandBit = 0x40000000u;          // set in bits(u' + e K) iff it is >= 2 (or NaN)

__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The exact Gumbel score z - ln(-ln u) of one entry (x its logit, w its Philox word).
__device__ __forceinline__ float gumbel_score(float x, uint32_t w, float invT)
{
    const float delta = (2.0f - u_prime(w)) - 5.9604644775390625e-8f;   // 1 - u, exact
    const float E = -log1pf(-delta);                                     // -ln u
    return x * invT - logf(E);
}

// A cheap estimate of the same score, within 2e-5 of it: ln E from lg2.approx, and -ln u from
// its series for 1 - u < 2^-5 (relative error < 8e-6), else from lg2.approx of u.  Both forms
// are computed and one is selected, so that the seed of a segment, where every entry of a batch
// takes it, runs without a branch.
__device__ __forceinline__ float gumbel_score_estimate_sel(float x, uint32_t w, float invT)
{
    const float delta = (2.0f - u_prime(w)) - 5.9604644775390625e-8f;
    const float Es = delta * fmaf(delta, fmaf(delta, 0.333333343f, 0.5f), 1.0f);
    const float El = -lg2_approx(1.0f - delta) * kLn2;
    return fmaf(-lg2_approx(delta < 0.03125f ? Es : El), kLn2, x * invT);
}

// The margin that covers the estimate's error and the rounding of either score near s.
__device__ __forceinline__ float estimate_margin(float s)
{
    return fmaf(fabsf(s), 9.5367431640625e-7f, 1.0e-4f);
}

__device__ __forceinline__ float cand_scale(float xm, float best, float c)
{
    return ex2(fmaf(xm, c, -best * kLog2e)) * kCandSlack;
}

__device__ __forceinline__ bool better(float s, int i, float bs, int bi)
{
    return s > bs || (s == bs && (unsigned)i < (unsigned)bi);
}

// Associative merge of two online states (c = log2(e) / T).
__device__ __forceinline__ void merge_state(RowState &a, float xm, float S, float T2, int ai,
                                            float best, int bi, float c)
{
    const float m = fmaxf(a.xm, xm);
    const float da = (a.xm - m) * c;
    const float db = (xm - m) * c;
    const float sa = ex2(da), sb = ex2(db);
    // a side whose weight underflows to 0 contributes nothing, even if its sums overflowed
    // (a slice holding only excluded entries far below the row maximum)
    const float T2n = (sa == 0.0f ? 0.0f : sa * fmaf(da, a.S, a.T2)) +
                      (sb == 0.0f ? 0.0f : sb * fmaf(db, S, T2));
    const float Sn = (sa == 0.0f ? 0.0f : a.S * sa) + (sb == 0.0f ? 0.0f : S * sb);
    int ain;
    if (a.xm > xm) ain = a.ai;
    else if (xm > a.xm) ain = ai;
    else ain = min(a.ai, ai);
    a.xm = m;
    a.S = Sn;
    a.T2 = T2n;
    a.ai = ain;
    if (better(best, bi, a.best, a.bi)) {
        a.best = best;
        a.bi = bi;
    }
}

__device__ __forceinline__ void warp_merge(RowState &st, float c)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float xm = __shfl_xor_sync(0xFFFFFFFFu, st.xm, off);
        const float S = __shfl_xor_sync(0xFFFFFFFFu, st.S, off);
        const float T2 = __shfl_xor_sync(0xFFFFFFFFu, st.T2, off);
        const int ai = __shfl_xor_sync(0xFFFFFFFFu, st.ai, off);
        const float best = __shfl_xor_sync(0xFFFFFFFFu, st.best, off);
        const int bi = __shfl_xor_sync(0xFFFFFFFFu, st.bi, off);
        merge_state(st, xm, S, T2, ai, best, bi, c);
    }
}

// Order-preserving unsigned key of a binary32 value (larger key = larger value; -0 and +0
// share +0's key; NaN takes key 0, below -inf, so that a maximum never picks it).
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f + 0.0f);
    return f != f ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The warp's best (score, index) by the order of better(): the largest score, then the lowest
// index (as unsigned, so -1 = none comes last), in two warp-wide reductions.
__device__ __forceinline__ void warp_best(float &best, int &bi)
{
    const uint32_t k = order_key(best);
    const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, k);
    const uint32_t imin = __reduce_min_sync(0xFFFFFFFFu, k == kmax ? (uint32_t)bi : 0xFFFFFFFFu);
    best = key_value(kmax);
    bi = (int)imin;
}

__device__ __forceinline__ RowState empty_state()
{
    return RowState{kEmptyMax, 0.0f, 0.0f, 0x7FFFFFFF, -INFINITY, -1};
}

// ---------------------------------------------------------------- e4m3 logits

// Four OCP e4m3 logits (byte i of w is entry i) as binary32.  Every e4m3 value, NaN included,
// is exact in binary16 and binary16 is exact in binary32, so both conversions are exact.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float &x0, float &x1, float &x2, float &x3)
{
    asm("{\n\t.reg .b16 q0, q1, h0, h1, h2, h3;\n\t.reg .b32 p01, p23;\n\t"
        "mov.b32 {q0, q1}, %4;\n\t"
        "cvt.rn.f16x2.e4m3x2 p01, q0;\n\t"
        "cvt.rn.f16x2.e4m3x2 p23, q1;\n\t"
        "mov.b32 {h0, h1}, p01;\n\t"
        "mov.b32 {h2, h3}, p23;\n\t"
        "cvt.f32.f16 %0, h0;\n\tcvt.f32.f16 %1, h1;\n\tcvt.f32.f16 %2, h2;\n\tcvt.f32.f16 %3, h3;\n\t}"
        : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3)
        : "r"(w));
}

// One e4m3 logit (the low byte of b) as binary32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b)
{
    float x0, x1, x2, x3;
    e4m3x4_to_f32(b & 0xFFu, x0, x1, x2, x3);
    return x0;
}

// ---------------------------------------------------------------- packed per-vector body

// Sums of one consumer thread over its part of a row, as two packed pairs each (four
// independent accumulation chains): S = sum 2^t, T2 = sum t 2^t.
struct PackedSums {
    f32x2 S0, S1, T0, T1;
};

__device__ __forceinline__ void packed_zero(PackedSums &q)
{
    q.S0 = q.S1 = q.T0 = q.T1 = 0ull;       // +0.0f in both halves
}

// New running maximum: every accumulator is rescaled by sc = 2^d (d <= 0).  A weight that
// underflows to 0 drops the old sums even if they overflowed.
__device__ __forceinline__ void packed_rescale(PackedSums &q, float d, float sc)
{
    if (sc == 0.0f) {
        packed_zero(q);
        return;
    }
    const f32x2 d2 = pk2(d, d), sc2 = pk2(sc, sc);
    q.T0 = mul2(sc2, fma2(d2, q.S0, q.T0));
    q.T1 = mul2(sc2, fma2(d2, q.S1, q.T1));
    q.S0 = mul2(q.S0, sc2);
    q.S1 = mul2(q.S1, sc2);
}

__device__ __forceinline__ void packed_fold(const PackedSums &q, RowState &st)
{
    float a, b, c, d;
    upk2(add2(q.S0, q.S1), a, b);
    upk2(add2(q.T0, q.T1), c, d);
    st.S = a + b;
    st.T2 = c + d;
}

// Philox4x32-10 with the round keys derived in place from the seed words (k0, k1).
__device__ __forceinline__ uint4 philox_seed(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                             uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128w(uint32_t addr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr)
                 : "memory");
    return r;
}

struct GumbelBest {
    float score;
    int idx;
};

// The rare exact pass over a group of N logits (entries v0 ..) whose candidate test passed:
// every entry with 1 - u < 2^t K takes the exact score z - ln(-ln u), and the best one so far
// is returned.  The caller passes the entries' Philox words (wa: entries 0-3, wb: 4-7), so
// nothing is drawn twice; 2^t is recomputed from the logits.  Kept out of line so that the
// unrolled hot loops stay small.
template <int N>
__device__ __noinline__ GumbelBest gumbel_exact_group(float4 xa, float4 xb, uint4 wa, uint4 wb, uint32_t v0,
                                                      float c, float invT, float nb, float K, GumbelBest best)
{
    const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    const uint32_t w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const float e = ex2(fmaf(x[j], c, nb));
        const float f = one_minus_u_plus(w[j]);
        if (f < fmaf(e, K, kCandAdd)) {
            const float delta = f - kOneMinusHalfUlp;          // 1 - u, exact
            const float E = -log1pf(-delta);                   // -ln u
            const float score = x[j] * invT - logf(E);
            const int idx = (int)(v0 + (uint32_t)j);
            if (better(score, idx, best.score, best.idx)) best = GumbelBest{score, idx};
        }
    }
    return best;
}

// The streaming kernel's exact pass over a group of N logits (entries v0 ..) of a lane whose
// candidate test passed.  The group's entries are tested again one by one (2^t recomputed from
// the logits exactly as the batch computed it) into a bit mask, and only the flagged entries,
// usually one, take the exact score, in a loop over the mask: the code stays small.
template <int N>
__device__ __noinline__ GumbelBest gumbel_exact_flagged(float4 xa, float4 xb, uint4 wa, uint4 wb, uint32_t v0,
                                                        float c, float invT, float nb, float K, GumbelBest best)
{
    const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    const uint32_t w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const float e = ex2(fmaf(x[j], c, nb));
        flags |= ((__float_as_uint(fmaf(e, K, u_prime(w[j]))) >> 30) & 1u) << j;
    }
#pragma unroll 1
    while (flags != 0u) {
        const int j = __ffs(flags) - 1;
        flags &= flags - 1u;
        float xj = x[0];
        uint32_t wj = w[0];
#pragma unroll
        for (int k = 1; k < N; ++k)
            if (j == k) {
                xj = x[k];
                wj = w[k];
            }
        const float score = gumbel_score(xj, wj, invT);
        const int idx = (int)(v0 + (uint32_t)j);
        if (better(score, idx, best.score, best.idx)) best = GumbelBest{score, idx};
    }
    return best;
}

// The same exact pass for callers that no longer hold the Philox words (the per-thread-row
// epilogue of the fused kernel, where keeping them live across the vote costs registers): the
// group's blocks are drawn again from the counter (v0 / 4, p, step, sw) and the seed words.
template <int N>
__device__ __noinline__ GumbelBest gumbel_exact_draw(float4 xa, float4 xb, uint32_t v0, float c, float invT,
                                                     float nb, float K, uint32_t p, uint32_t step, uint32_t sw,
                                                     uint32_t k0, uint32_t k1, GumbelBest best)
{
    const uint4 wa = philox_seed(v0 >> 2, p, step, sw, k0, k1);
    const uint4 wb = N == 8 ? philox_seed((v0 >> 2) + 1, p, step, sw, k0, k1) : make_uint4(0u, 0u, 0u, 0u);
    return gumbel_exact_group<N>(xa, xb, wa, wb, v0, c, invT, nb, K, best);
}

// Per-row values of the arithmetic: c = log2(e) / T and 1 / T of the row's canvas, the
// canvas's step and the row's Philox counter words (position p, stream and canvas id sw).
struct RowCtx {
    float c, invT;
    uint32_t step, p, sw;
};

// N = 8 or 4 consecutive logits x of a canvas row, entries v0 .. v0+N-1 (v0 a multiple of
// N): running max / first argmax, S and T2 (on packed f32x2 pairs), and
// for masked rows the per-entry Gumbel candidate test 1 - u < 2^t K, whose rare passes take
// the exact score.  `a` supplies c = log2(e)/T, invT = 1/T, the step and the Philox round
// keys.  WARP_ROW: the 32 lanes work on the same row (they share the best score when it
// moves, so every lane must call this with the same trip count; `valid` masks lanes without a
// group); otherwise every lane owns its row.  `gumbel` (runtime) switches the sampling part
// off for a lane whose row is not masked.  `stash` (per-thread rows only) is the shared address
// of a 32-byte slot of this thread that keeps a candidate group's Philox words for the exact
// pass; with WARP_ROW the pass draws them again.
template <int N, bool MASKED, bool WARP_ROW, typename Args>
__device__ __forceinline__ void consume_vals(const float (&x)[N], bool valid, uint32_t v0, const Args &a,
                                             const RowCtx &rc, f32x2 c2, RowState &st,
                                             PackedSums &q, float &nb, f32x2 &nb2, float &K,
                                             bool gumbel = true, uint32_t stash = 0u)
{
    float vmax = 0.0f;
    float e[N];
    if (valid) {
        if constexpr (N == 8) vmax = max3(max3(x[0], x[1], x[2]), max3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
        else vmax = max3(x[0], x[1], fmaxf(x[2], x[3]));
    }
    // a new running maximum is rare after the first groups; the vote keeps this a real branch
    // (the compiler would otherwise predicate the whole block into every group)
    const bool newmax = valid && vmax > st.xm;
    if constexpr (WARP_ROW) {
        // the lanes share one running maximum (the reference of every lane's sums), so a new
        // maximum is a record of the whole warp's part of the row, not of each lane's
        if (__any_sync(0xFFFFFFFFu, newmax)) {
            float wm = valid ? vmax : -INFINITY;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
            // first entry holding it: entries grow with the lane within one group of vectors
            int idx = 0x7FFFFFFF;
            if (valid && vmax == wm) {
                int j0 = N - 1;
#pragma unroll
                for (int j = N - 1; j >= 0; --j)
                    if (x[j] == wm) j0 = j;
                idx = (int)(v0 + (uint32_t)j0);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, off));
            const float d = (st.xm - wm) * rc.c;
            packed_rescale(q, d, ex2(d));
            st.ai = idx;
            st.xm = wm;
            nb = -wm * rc.c;
            nb2 = pk2(nb, nb);
            if (MASKED && gumbel) K = cand_scale(st.xm, st.best, rc.c);
        }
    } else if (__any_sync(__activemask(), newmax)) {
        if (newmax) {
                const float d = (st.xm - vmax) * rc.c;
                packed_rescale(q, d, ex2(d));
                int j0 = N - 1;
#pragma unroll
                for (int j = N - 1; j >= 0; --j)
                    if (x[j] == vmax) j0 = j;
                st.ai = (int)(v0 + (uint32_t)j0);
                st.xm = vmax;
                nb = -vmax * rc.c;
                nb2 = pk2(nb, nb);
            if (MASKED && gumbel) K = cand_scale(st.xm, st.best, rc.c);
        }
    }
    if (valid) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const f32x2 tp = fma2(pk2(x[2 * i], x[2 * i + 1]), c2, nb2);
            float t0, t1;
            upk2(tp, t0, t1);
            e[2 * i] = ex2(t0);
            e[2 * i + 1] = ex2(t1);
            const f32x2 ep = pk2(e[2 * i], e[2 * i + 1]);
            if (i & 1) {
                q.S1 = add2(q.S1, ep);
                q.T1 = fma2(tp, ep, q.T1);
            } else {
                q.S0 = add2(q.S0, ep);
                q.T0 = fma2(tp, ep, q.T0);
            }
        }
    }
    if constexpr (MASKED) {
        bool cand = false;
        if (valid && gumbel) {
            const uint4 u0 = philox(v0 >> 2, rc.p, rc.step, rc.sw, a.keys);
            uint4 u1 = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (N == 8) u1 = philox((v0 >> 2) + 1, rc.p, rc.step, rc.sw, a.keys);
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int j = 0; j < N; ++j) cand |= one_minus_u_plus(w[j]) < fmaf(e[j], K, kCandAdd);
            // a candidate's words go to the thread's shared slot, so that they need not stay
            // live in registers across the vote nor be drawn again
            if (!WARP_ROW && cand) {
                sts128(stash, u0);
                sts128(stash + 16u, u1);
            }
        }
        const bool go = __any_sync(WARP_ROW ? 0xFFFFFFFFu : __activemask(), cand);
        if (go) {
            if (cand) {
                const float4 xa = make_float4(x[0], x[1], x[2], x[3]);
                const float4 xb = N == 8 ? make_float4(x[N > 4 ? 4 : 0], x[N > 5 ? 5 : 0], x[N > 6 ? 6 : 0],
                                                       x[N > 7 ? 7 : 0])
                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                GumbelBest g;
                if constexpr (!WARP_ROW)
                    g = gumbel_exact_group<N>(xa, xb, lds128w(stash), lds128w(stash + 16u), v0, rc.c, rc.invT, nb, K,
                                              GumbelBest{st.best, st.bi});
                else
                    g = gumbel_exact_draw<N>(xa, xb, v0, rc.c, rc.invT, nb, K, rc.p, rc.step, rc.sw, a.keys.k[0],
                                             a.keys.k[1], GumbelBest{st.best, st.bi});
                st.best = g.score;
                st.bi = g.idx;
            }
            if (WARP_ROW) warp_best(st.best, st.bi);
            K = cand_scale(st.xm, st.best, rc.c);
        }
    }
}

// One 16-byte vector of VEC logits (8 bf16 or 4 fp32) of a row, entries jvec*VEC ..
template <int VEC, bool MASKED>
__device__ __forceinline__ void consume_packed(const uint4 r, bool valid, uint32_t jvec, const K1Args &a,
                                               const RowCtx &rc, f32x2 c2, RowState &st,
                                               PackedSums &q, float &nb, f32x2 &nb2, float &K,
                                               bool gumbel = true)
{
    static_assert(VEC == 4 || VEC == 8, "e4m3 tails go through consume_vals in half vectors");
    {
        float x[VEC];
        if constexpr (VEC == 8) {
            const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = __uint_as_float(w4[i] << 16);
                x[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
            }
        } else {
            x[0] = __uint_as_float(r.x);
            x[1] = __uint_as_float(r.y);
            x[2] = __uint_as_float(r.z);
            x[3] = __uint_as_float(r.w);
        }
        consume_vals<VEC, MASKED, true>(x, valid, jvec * VEC, a, rc, c2, st, q, nb, nb2, K, gumbel);
    }
}

// Largest of N floats (N = 4, 8, 16 or 32) with three-input maxima.
template <int N>
__device__ __forceinline__ float vec_max(const float (&x)[N])
{
    if constexpr (N == 4) {
        return max3(x[0], x[1], fmaxf(x[2], x[3]));
    } else if constexpr (N == 8) {
        return max3(max3(x[0], x[1], x[2]), max3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
    } else if constexpr (N == 16) {
        const float m0 = max3(x[0], x[1], x[2]), m1 = max3(x[3], x[4], x[5]), m2 = max3(x[6], x[7], x[8]);
        const float m3 = max3(x[9], x[10], x[11]), m4 = max3(x[12], x[13], x[14]);
        return max3(max3(m0, m1, m2), m3, fmaxf(m4, x[15]));
    } else {
        static_assert(N == 32, "vec_max: N is 4, 8, 16 or 32");
        float m[11];
#pragma unroll
        for (int i = 0; i < 10; ++i) m[i] = max3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
        m[10] = fmaxf(x[30], x[31]);
        return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), max3(max3(m[6], m[7], m[8]), m[9], m[10]));
    }
}

// U whole vectors of one lane of a warp that streams one row: vector u holds the VEC entries
// from (jv0 + 32 u) VEC on.  The arithmetic per entry is that of consume_vals (the warp shares
// one running maximum and one best Gumbel score), but a whole batch takes one new-maximum vote
// and, for a masked row, one candidate vote.  The Philox blocks of all U vectors are drawn
// after the new-maximum vote, in the same basic block as the exponentials and the sums, so
// that their independent chains overlap with the rest.
template <int VEC, int U, bool MASKED>
__device__ __forceinline__ void consume_batch(const uint4 (&r)[U], uint32_t jv0, const K1Args &a, const RowCtx &rc,
                                              const PhiloxRow &ph, f32x2 c2, RowState &st, PackedSums &q,
                                              float &nb, f32x2 &nb2, float &K, float &bt)
{
    constexpr int N = U * VEC;
    float x[N];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if constexpr (VEC == 16) {
            e4m3x4_to_f32(r[u].x, x[16 * u + 0], x[16 * u + 1], x[16 * u + 2], x[16 * u + 3]);
            e4m3x4_to_f32(r[u].y, x[16 * u + 4], x[16 * u + 5], x[16 * u + 6], x[16 * u + 7]);
            e4m3x4_to_f32(r[u].z, x[16 * u + 8], x[16 * u + 9], x[16 * u + 10], x[16 * u + 11]);
            e4m3x4_to_f32(r[u].w, x[16 * u + 12], x[16 * u + 13], x[16 * u + 14], x[16 * u + 15]);
        } else if constexpr (VEC == 8) {
            const uint32_t w4[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[8 * u + 2 * i] = __uint_as_float(w4[i] << 16);
                x[8 * u + 2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
            }
        } else {
            x[4 * u + 0] = __uint_as_float(r[u].x);
            x[4 * u + 1] = __uint_as_float(r[u].y);
            x[4 * u + 2] = __uint_as_float(r[u].z);
            x[4 * u + 3] = __uint_as_float(r[u].w);
        }
    }
    const float vmax = vec_max<N>(x);
    if (__any_sync(0xFFFFFFFFu, vmax > st.xm)) {
        const float wm = key_value(__reduce_max_sync(0xFFFFFFFFu, order_key(vmax)));
        // first entry holding it: this lane's entries grow with the vector, then the entry, and
        // all of the warp's vector u precede its vector u + 1
        uint32_t idx = 0x7FFFFFFFu;
        if (vmax == wm) {
#pragma unroll
            for (int i = N - 1; i >= 0; --i)
                if (x[i] == wm) idx = (jv0 + 32u * (uint32_t)(i / VEC)) * (uint32_t)VEC + (uint32_t)(i % VEC);
        }
        idx = __reduce_min_sync(0xFFFFFFFFu, idx);
        const float d = (st.xm - wm) * rc.c;
        packed_rescale(q, d, ex2(d));
        st.ai = idx;
        st.xm = wm;
        nb = -wm * rc.c;
        nb2 = pk2(nb, nb);
        if constexpr (MASKED) K = cand_scale(st.xm, fmaxf(st.best, bt), rc.c);
    }
    // the Philox words of the batch's entries (masked rows), drawn after the vote so that they
    // are not live across its branch; their chains interleave with the exponentials below
    uint32_t w[MASKED ? N : 1];
    if constexpr (MASKED) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int k = 0; k < VEC / 4; ++k) {
                const uint4 g = philox_row_block((jv0 + 32u * (uint32_t)u) * (uint32_t)(VEC / 4) + (uint32_t)k, ph,
                                                 a.keys);
                w[VEC * u + 4 * k + 0] = g.x;
                w[VEC * u + 4 * k + 1] = g.y;
                w[VEC * u + 4 * k + 2] = g.z;
                w[VEC * u + 4 * k + 3] = g.w;
            }
    }
    float e[N];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const f32x2 tp = fma2(pk2(x[2 * i], x[2 * i + 1]), c2, nb2);
        float t0, t1;
        upk2(tp, t0, t1);
        e[2 * i] = ex2(t0);
        e[2 * i + 1] = ex2(t1);
        const f32x2 ep = pk2(e[2 * i], e[2 * i + 1]);
        if (i & 1) {
            q.S1 = add2(q.S1, ep);
            q.T1 = fma2(tp, ep, q.T1);
        } else {
            q.S0 = add2(q.S0, ep);
            q.T0 = fma2(tp, ep, q.T0);
        }
    }
    if constexpr (MASKED) {
        if (bt == -INFINITY) {
            // the segment's first batch: the largest score estimate of all its entries, less the
            // estimate's margin, is a lower bound of the segment's best score.  With it as the
            // threshold, only entries near that maximum pass the candidate test below.
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < N; ++i) m = fmaxf(m, gumbel_score_estimate_sel(x[i], w[i], rc.invT));
            m = key_value(__reduce_max_sync(0xFFFFFFFFu, order_key(m)));
            bt = m == INFINITY ? m : m - estimate_margin(m);
            K = cand_scale(st.xm, fmaxf(st.best, bt), rc.c);
        }
        // candidate test of two entries at a time: u' + 2^t K on packed FMA, the results' bits
        // or-ed together; bit 30 of the or is set iff some entry's sum reached 2
        uint32_t cacc[U];
        const f32x2 K2 = pk2(K, K);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            cacc[u] = 0u;
#pragma unroll
            for (int j = 0; j < VEC; j += 2) {
                float d0, d1;
                upk2(fma2(pk2(e[VEC * u + j], e[VEC * u + j + 1]), K2,
                          pk2(u_prime(w[VEC * u + j]), u_prime(w[VEC * u + j + 1]))), d0, d1);
                cacc[u] |= __float_as_uint(d0) | __float_as_uint(d1);
            }
        }
        bool cand[U];
        bool any = false;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            cand[u] = (cacc[u] & kCandBit) != 0u;
            any |= cand[u];
        }
        if (__any_sync(0xFFFFFFFFu, any)) {
            // the exact pass takes groups of up to 8 entries (two per e4m3 vector)
            constexpr int G8 = VEC < 8 ? VEC : 8;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (cand[u]) {
#pragma unroll
                    for (int h = 0; h < VEC / G8; ++h) {
                        const int o = VEC * u + G8 * h;
                        const float4 xa = make_float4(x[o], x[o + 1], x[o + 2], x[o + 3]);
                        const float4 xb = G8 == 8 ? make_float4(x[o + (G8 > 4 ? 4 : 0)], x[o + (G8 > 5 ? 5 : 0)],
                                                                x[o + (G8 > 6 ? 6 : 0)], x[o + (G8 > 7 ? 7 : 0)])
                                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        const uint4 wa = make_uint4(w[o], w[o + 1], w[o + 2], w[o + 3]);
                        const uint4 wb = G8 == 8 ? make_uint4(w[o + (G8 > 4 ? 4 : 0)], w[o + (G8 > 5 ? 5 : 0)],
                                                              w[o + (G8 > 6 ? 6 : 0)], w[o + (G8 > 7 ? 7 : 0)])
                                                 : make_uint4(0u, 0u, 0u, 0u);
                        const GumbelBest g = gumbel_exact_flagged<G8>(
                            xa, xb, wa, wb, (jv0 + 32u * (uint32_t)u) * (uint32_t)VEC + (uint32_t)(G8 * h), rc.c, rc.invT,
                            nb, K, GumbelBest{st.best, st.bi});
                        st.best = g.score;
                        st.bi = g.idx;
                    }
                }
            warp_best(st.best, st.bi);
            K = cand_scale(st.xm, fmaxf(st.best, bt), rc.c);
        }
    }
}

// ---------------------------------------------------------------- mbarrier / bulk copy PTX

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Waits until the barrier's phase with parity `parity` has completed; false after `limit`
// unsuccessful polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit = kWaitLimit)
{
    const uint32_t a = smem_addr(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// ---------------------------------------------------------------- row partition

// Weight-space prefix P[r] of row r (weighted mode: from shared memory; uniform mode:
// every row weighs nvec_row).
struct Partition {
    const uint32_t *P;      // shared, [rows + 1], weighted mode only
    long long nvec;
    int rows;
    int weighted;
    __device__ __forceinline__ unsigned long long start(int r) const
    {
        return weighted ? (unsigned long long)P[r] : (unsigned long long)r * (unsigned long long)nvec;
    }
    __device__ __forceinline__ unsigned long long total() const { return start(rows); }
    // first row whose weight range ends after w
    __device__ __forceinline__ int first_row_after(unsigned long long w) const
    {
        if (!weighted) return (int)(w / (unsigned long long)nvec);
        int lo = 0, hi = rows;   // smallest r in [0, rows] with P[r + 1] > w
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((unsigned long long)P[mid + 1] > w) hi = mid;
            else lo = mid + 1;
        }
        return lo;
    }
};

// The row segments of CTA `cta`: every row whose weight range meets [lo, hi), with the
// vector range [j0, j1) of the vectors whose weight offsets start inside [lo, hi).
struct SegmentCursor {
    Partition part;
    unsigned long long lo, hi;
    int r;
    __device__ __forceinline__ void begin(const Partition &p, int cta, int G)
    {
        part = p;
        const unsigned long long W = p.total();
        lo = (unsigned long long)cta * W / (unsigned long long)G;
        hi = (unsigned long long)(cta + 1) * W / (unsigned long long)G;
        r = (lo < hi) ? p.first_row_after(lo) : p.rows;
    }
    // next segment; false when done.  Rows of zero weight are skipped.  `first` / `last`: the
    // segment starts / ends the row's weight range (so this unit is the row's first / last).
    bool first = false, last = false;
    __device__ __forceinline__ bool next(int &row, long long &j0, long long &j1)
    {
        while (r < part.rows) {
            const unsigned long long a = part.start(r), b = part.start(r + 1);
            if (a >= hi) {
                r = part.rows;
                return false;
            }
            const int cur = r++;
            if (b == a) continue;
            const unsigned long long wv = (b - a) / (unsigned long long)part.nvec;
            const unsigned long long s0 = (lo > a ? lo : a) - a;
            const unsigned long long s1 = (hi < b ? hi : b) - a;
            row = cur;
            j0 = (long long)((s0 + wv - 1) / wv);
            j1 = (long long)((s1 + wv - 1) / wv);
            if (j1 > part.nvec) j1 = part.nvec;
            if (j0 > j1) j0 = j1;
            first = a >= lo;       // this unit holds the row's first weight unit
            last = b <= hi;        // ... and its last one
            return true;
        }
        return false;
    }
};

}  // namespace ebk
