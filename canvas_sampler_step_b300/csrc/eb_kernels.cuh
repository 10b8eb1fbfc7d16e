// eb_kernels.cuh -- device code of the B300 (sm_103a) Entropy-Bounded (EB) denoising sampler
// step of DiffusionGemma (model card, "Best practices" section 1, "Diffusion sampling
// settings": at most 48 steps, temperature 0.8 -> 0.4 for logit shaping, lowest-entropy
// selection under the entropy bound 0.1, full re-noising of the unselected tokens, adaptive
// stop at mean entropy < 0.005 with an argmax stable over two consecutive steps).
//
// k1_rowstats (one launch per step) streams the [B, L, V] logits exactly once.
//   * Work split.  Row r of a running canvas weighs nvec * w (w = w_masked for masked rows,
//     which also draw Gumbel noise, w_unmasked otherwise; rows of halted canvases weigh 0).
//     The prefix sums P of the weights are cut into G equal ranges, one per CTA (G = one CTA
//     per SM), so CTAs finish together even though masked rows cost more instructions per
//     byte, and halted canvases cost nothing.  CTA c writes one partial state for every row
//     its range touches to slot (row + c) of the workspace (the (row, CTA) pairs form a
//     staircase, so row + c is unique).
//   * Data movement.  One producer warp moves the CTA's rows through a ring of 16 KiB
//     shared-memory stages with 1-D TMA bulk copies (cp.async.bulk ... mbarrier::complete_tx);
//     16 consumer warps read 16-byte vectors from shared memory.  Every mbarrier wait is
//     bounded; a CTA whose wait gives up marks its partials and returns.
//   * Per element: t = x * log2(e)/T - xm * log2(e)/T, e = 2^t (MUFU), S += e, T2 += t e,
//     with xm the running maximum of the thread's raw logits (first index kept for the
//     argmax).  H = ln 2 (log2 S - T2 / S) after merging.
//   * Gumbel-max for masked rows: with u from a Philox4x32-10 word and E = -ln u, the sample
//     maximises z - ln E.  Since E >= 1 - u, an entry can beat the best score so far only if
//     1 - u < 2^t K, K = 2^(xm log2e / T - best log2e); that test is one LOP3, one FFMA and
//     one predicate-or per entry.  Entries that pass it (a handful per warp and row) take the
//     exact score z - logf(-log1pf(-(1 - u))); the warp shares its best score when it moves.
// k2_select (one CTA per canvas) merges each row's partials in ascending CTA order
// (deterministic), runs the stop test, the entropy-bounded selection and the commit /
// re-mask / finalisation.  Sums of entropies are exact 64-bit fixed point (2^-40 nats).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "eb_sampler.h"

namespace ebk {

// ---------------------------------------------------------------- launch geometry
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kK1Threads = kConsumers + 32;        // + one producer warp
constexpr int kVecPerStage = 1024;                  // 16-byte vectors per ring stage
constexpr int kStageBytes = kVecPerStage * 16;
constexpr int kStages = 10;
constexpr int kMaxWeightedRows = 4096;
constexpr int kK2Threads = 256;
constexpr int kMaxL = 1024;
constexpr int kMaxGrid = 8192;
constexpr int kWeightUnmasked = 4;
constexpr int kWeightMasked = 10;
constexpr uint32_t kWaitLimit = 1u << 26;           // mbarrier polls before giving up

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

struct K1Args {
    const void *logits;
    const uint8_t *mask;
    const int32_t *status;
    Partial *partials;
    uint32_t *prefix_out;   // [rows + 1] weight prefix (weighted mode; written by CTA 0)
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
};

struct K2Args {
    const Partial *partials;
    const uint32_t *prefix;  // weighted mode: [rows + 1]
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
    int k3_g;                  // > 0: partials come from the fused unembedding kernel, whose
                               // row block mb, group rank j < k3_g and column half hh write
                               // slot ((mb k3_g + j) 2 + hh) 128 + row % 128
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

// f = 1 + (0x7FFFFF - j) 2^-23 for j = low 23 bits of w, so that 1 - u = f - (1 - 2^-24)
// exactly, u = (j + 1/2) 2^-23 being the entry's uniform.
__device__ __forceinline__ float one_minus_u_plus(uint32_t w)
{
    return __uint_as_float((w & 0x7FFFFFu) ^ 0x3FFFFFFFu);
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

__device__ __forceinline__ void warp_best(float &best, int &bi)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
        if (better(ob, oi, best, bi)) {
            best = ob;
            bi = oi;
        }
    }
}

__device__ __forceinline__ RowState empty_state()
{
    return RowState{kEmptyMax, 0.0f, 0.0f, 0x7FFFFFFF, -INFINITY, -1};
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

// Waits until the barrier's phase with parity `parity` has completed; false after kWaitLimit
// unsuccessful polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
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

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
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
    // next segment; false when done.  Rows of zero weight are skipped.
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
            return true;
        }
        return false;
    }
};

}  // namespace ebk
