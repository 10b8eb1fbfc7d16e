// eb_sampler.cu -- B300 (sm_103a) kernels and C ABI of the Entropy-Bounded (EB) denoising
// sampler step of DiffusionGemma (model card, "Best practices" section 1, "Diffusion
// sampling settings": 48 steps, temperature 0.8 -> 0.4 for logit shaping, lowest-entropy
// selection under the entropy bound 0.1, full re-noising of the unselected tokens,
// adaptive stop at mean entropy < 0.005 with an argmax stable over two steps).
//
// Two kernels per step:
//   k1_rowstats  streams the [B, L, V] logits once.  The flattened (row, 16-byte vector)
//                index space is cut into G equal contiguous ranges, one per CTA (G = SMs x
//                resident CTAs), so every CTA moves the same number of bytes.  Each thread
//                keeps an online state per row segment: the running raw max xm and its first
//                index, S = sum 2^t and T2 = sum t 2^t with t = (x - xm) log2(e) / T, and for
//                masked rows the best Gumbel score.  A CTA writes one partial state per row
//                segment it touched to slot (row + cta) of the workspace.
//   k2_select    one CTA per canvas: merges the partials of its rows in a fixed order
//                (deterministic), forms H = ln2 (log2 S - T2 / S), runs the stop test, the
//                entropy-bounded selection (bitonic sort of (H, position) keys, prefix sums
//                in binary64), commits / re-masks and finalises complete / capped canvases.
//
// Gumbel-max without a log per entry: with E_v = -ln u_v the sample is the v maximising
// z_v - ln E_v.  Since E_v >= delta_v = 1 - u_v (exact from the Philox word), an entry can
// only beat the current best score `best` if delta_v < 2^t_v * 2^(xm log2e / T - best
// log2e).  That test costs one multiply and compare per entry; only entries that pass it
// (a handful per warp and row) evaluate the exact score with log1pf / logf.  The best score
// is shared across the warp whenever it improves, which keeps the pass rate low.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "eb_sampler.h"

namespace ebk {

constexpr int kK1Threads = 256;
constexpr int kK1Unroll = 4;
constexpr int kK2Threads = 256;
constexpr int kMaxL = 1024;
constexpr int kMaxGrid = 8192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kEmptyMax = -1.0e30f;     // running max of a slice that saw no element
constexpr float kMinT = -16384.0f;        // log2-domain clamp: 2^t is exactly 0 below it
constexpr float kCandSlack = 1.0f + 1.0f / 256.0f;
constexpr float kOneMinusHalfUlp = 0.99999994039535522f;  // 1 - 2^-24
constexpr uint32_t kStreamGumbel = 1u;

// Philox4x32-10 round keys (k0 + r * 0x9E3779B9, k1 + r * 0xBB67AE85), r = 0..9; computed
// on the host and passed as a kernel parameter so that each xor reads the constant bank.
struct RoundKeys {
    uint32_t k[20];
};

// Per-(row, CTA) partial state.  xm: max raw logit of the slice (kEmptyMax if empty);
// S, T2: sums of 2^t and t 2^t, t = (x - xm) c, c = log2(e) / T; ai: first index of xm;
// best / bi: best Gumbel score z - ln E and its index (-inf / -1 if none).
struct __align__(16) Partial {
    float xm, S, T2;
    int ai;
    float best;
    int bi;
    int pad0, pad1;
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
    long long nvec_row;  // vectors (16 B, or 1 element on the scalar path) per row
    long long N;         // rows * nvec_row
    int L;
    int G;
    int step;
    float c;             // log2(e) / T
    float invT;          // 1 / T
    RoundKeys keys;
};

struct K2Args {
    const Partial *partials;
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
    long long N;
    int L;
    int G;
    int step;
    int max_steps;
    float c;
    float bound;
    float stop_entropy;
};

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Philox4x32-10 (Salmon et al., SC'11): two 32x32->64 products per round, high halves
// xored with the other counter words and the round key.
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

// delta = 1 - u for the uniform u = (j + 1/2) 2^-23, j = low 23 bits of w; exact.
__device__ __forceinline__ float gumbel_delta(uint32_t w)
{
    return __uint_as_float((w & 0x7FFFFFu) ^ 0x3FFFFFFFu) - kOneMinusHalfUlp;
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
    const float T2n = sa * fmaf(da, a.S, a.T2) + sb * fmaf(db, S, T2);
    const float Sn = a.S * sa + S * sb;
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

// ------------------------------------------------------------------ element kinds

enum Kind { kF32Vec = 0, kBF16Vec = 1, kF32Scalar = 2, kBF16Scalar = 3 };

template <int KIND> struct KindTraits;
template <> struct KindTraits<kF32Vec> {
    static constexpr int VEC = 4;
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const void *row, long long i)
    {
        return ldg_stream(reinterpret_cast<const uint4 *>(row) + i);
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[4])
    {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
};
template <> struct KindTraits<kBF16Vec> {
    static constexpr int VEC = 8;
    using Raw = uint4;
    static __device__ __forceinline__ Raw load(const void *row, long long i)
    {
        return ldg_stream(reinterpret_cast<const uint4 *>(row) + i);
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[8])
    {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xFFFF0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        x[4] = __uint_as_float(r.z << 16);
        x[5] = __uint_as_float(r.z & 0xFFFF0000u);
        x[6] = __uint_as_float(r.w << 16);
        x[7] = __uint_as_float(r.w & 0xFFFF0000u);
    }
};
template <> struct KindTraits<kF32Scalar> {
    static constexpr int VEC = 1;
    using Raw = float;
    static __device__ __forceinline__ Raw load(const void *row, long long i)
    {
        return __ldg(reinterpret_cast<const float *>(row) + i);
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[1]) { x[0] = r; }
};
template <> struct KindTraits<kBF16Scalar> {
    static constexpr int VEC = 1;
    using Raw = unsigned short;
    static __device__ __forceinline__ Raw load(const void *row, long long i)
    {
        return __ldg(reinterpret_cast<const unsigned short *>(row) + i);
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[1])
    {
        x[0] = __uint_as_float((uint32_t)r << 16);
    }
};

template <int KIND> __host__ __device__ constexpr int elem_bytes()
{
    return (KIND == kF32Vec || KIND == kF32Scalar) ? 4 : 2;
}

// Philox words of the VEC entries starting at vector index i (entry v0 = i * VEC).
template <int VEC>
__device__ __forceinline__ void gumbel_words(long long i, uint32_t p, uint32_t s, uint32_t sw,
                                             const RoundKeys &K, uint32_t (&w)[VEC])
{
    if constexpr (VEC == 8) {
        const uint4 a = philox((uint32_t)(2 * i), p, s, sw, K);
        const uint4 b = philox((uint32_t)(2 * i + 1), p, s, sw, K);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (VEC == 4) {
        const uint4 a = philox((uint32_t)i, p, s, sw, K);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else {
        const uint4 a = philox((uint32_t)(i >> 2), p, s, sw, K);
        const uint32_t q = (uint32_t)(i & 3);
        w[0] = q == 0 ? a.x : (q == 1 ? a.y : (q == 2 ? a.z : a.w));
    }
}

// One row segment [i0, i1) (vector indices within row r) by the whole CTA.
template <int KIND, bool MASKED>
__device__ __forceinline__ void k1_segment_loop(const K1Args &a, const void *rowp, long long i0,
                                                long long i1, uint32_t p, uint32_t sw,
                                                RowState &st)
{
    using T = KindTraits<KIND>;
    constexpr int VEC = T::VEC;
    const int tid = threadIdx.x;
    float nb = -st.xm * a.c;
    float K = MASKED ? cand_scale(st.xm, st.best, a.c) : 0.0f;
    for (long long base = i0; base < i1; base += (long long)kK1Threads * kK1Unroll) {
        typename T::Raw raw[kK1Unroll];
        bool valid[kK1Unroll];
#pragma unroll
        for (int u = 0; u < kK1Unroll; ++u) {
            const long long i = base + (long long)u * kK1Threads + tid;
            valid[u] = i < i1;
            if (valid[u]) raw[u] = T::load(rowp, i);
        }
#pragma unroll
        for (int u = 0; u < kK1Unroll; ++u) {
            const long long i = base + (long long)u * kK1Threads + tid;
            float x[VEC];
            float e[VEC];
            if (valid[u]) {
                T::unpack(raw[u], x);
                float vmax = x[0];
#pragma unroll
                for (int j = 1; j < VEC; ++j) vmax = fmaxf(vmax, x[j]);
                if (vmax > st.xm) {
                    const float d = (st.xm - vmax) * a.c;
                    const float sc = ex2(d);
                    st.T2 = sc * fmaf(d, st.S, st.T2);
                    st.S *= sc;
                    int j0 = VEC - 1;
#pragma unroll
                    for (int j = VEC - 1; j >= 0; --j)
                        if (x[j] == vmax) j0 = j;
                    st.ai = (int)(i * VEC + j0);
                    st.xm = vmax;
                    nb = -vmax * a.c;
                    if (MASKED) K = cand_scale(st.xm, st.best, a.c);
                }
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float t = fmaxf(fmaf(x[j], a.c, nb), kMinT);
                    e[j] = ex2(t);
                    st.S += e[j];
                    st.T2 = fmaf(t, e[j], st.T2);
                }
            }
            if constexpr (MASKED) {
                uint32_t cand = 0;
                uint32_t w[VEC];
                if (valid[u]) {
                    gumbel_words<VEC>(i, p, (uint32_t)a.step, sw, a.keys, w);
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        if (e[j] * K > gumbel_delta(w[j])) cand |= 1u << j;
                }
                if (__any_sync(0xFFFFFFFFu, cand != 0)) {
                    while (cand) {
                        const int j = __ffs(cand) - 1;
                        cand &= cand - 1;
                        float xj = x[0];
                        uint32_t wj = w[0];
#pragma unroll
                        for (int q = 1; q < VEC; ++q)
                            if (q == j) { xj = x[q]; wj = w[q]; }
                        const float E = -log1pf(-gumbel_delta(wj));
                        const float score = xj * a.invT - logf(E);
                        const int idx = (int)(i * VEC + j);
                        if (better(score, idx, st.best, st.bi)) {
                            st.best = score;
                            st.bi = idx;
                        }
                    }
                    warp_best(st.best, st.bi);
                    K = cand_scale(st.xm, st.best, a.c);
                }
            }
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(kK1Threads) k1_rowstats(const K1Args a)
{
    using T = KindTraits<KIND>;
    __shared__ RowState red[kK1Threads / 32];
    const int cta = blockIdx.x;
    const long long lo = (long long)cta * a.N / a.G;
    const long long hi = (long long)(cta + 1) * a.N / a.G;
    const size_t row_bytes = (size_t)a.nvec_row * T::VEC * elem_bytes<KIND>();
    long long seg = lo;
    while (seg < hi) {
        const long long r = seg / a.nvec_row;
        const long long rend = min(hi, (r + 1) * a.nvec_row);
        const long long i0 = seg - r * a.nvec_row;
        const long long i1 = rend - r * a.nvec_row;
        seg = rend;
        const int b = (int)(r / a.L);
        const uint32_t p = (uint32_t)(r - (long long)b * a.L);
        if (a.status[b] != EB_RUNNING) continue;   // CTA-uniform
        const bool masked = a.mask[r] != 0;
        const void *rowp = static_cast<const char *>(a.logits) + (size_t)r * row_bytes;
        const uint32_t sw = (kStreamGumbel << 24) | (uint32_t)b;
        RowState st{kEmptyMax, 0.0f, 0.0f, 0, -INFINITY, -1};
        if (masked) k1_segment_loop<KIND, true>(a, rowp, i0, i1, p, sw, st);
        else k1_segment_loop<KIND, false>(a, rowp, i0, i1, p, sw, st);
        warp_merge(st, a.c);
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 0) red[warp] = st;
        __syncthreads();
        if (warp == 0) {
            RowState s2 = lane < kK1Threads / 32 ? red[lane]
                                                 : RowState{kEmptyMax, 0.0f, 0.0f, 0x7FFFFFFF,
                                                            -INFINITY, -1};
            warp_merge(s2, a.c);
            if (lane == 0) {
                Partial out;
                out.xm = s2.xm;
                out.S = s2.S;
                out.T2 = s2.T2;
                out.ai = s2.ai;
                out.best = s2.best;
                out.bi = s2.bi;
                out.pad0 = 0;
                out.pad1 = 0;
                a.partials[r + cta] = out;
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ selection kernel

__device__ __forceinline__ long long range_start(long long c, long long N, int G)
{
    return c * N / G;
}

__device__ __forceinline__ int cta_of(long long i, long long N, int G)
{
    return (int)(((i + 1) * (long long)G - 1) / N);
}

__device__ double block_sum_double(double v, double *scratch)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += scratch[w];
        scratch[32] = t;
    }
    __syncthreads();
    return scratch[32];
}

__global__ void __launch_bounds__(kK2Threads) k2_select(const K2Args a)
{
    __shared__ float Hs[kMaxL];
    __shared__ int As[kMaxL];
    __shared__ int Ys[kMaxL];
    __shared__ unsigned long long keys[kMaxL];
    __shared__ double scan[kMaxL];
    __shared__ double red[33];
    __shared__ int counts[2];   // [0] committed this step, [1] masked before selection

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int L = a.L;
    if (a.status[b] != EB_RUNNING) return;   // CTA-uniform
    const long long rowbase = (long long)b * L;
    if (tid == 0) {
        counts[0] = 0;
        counts[1] = 0;
    }

    // 1. merge the per-CTA partials of every row in ascending CTA order (deterministic)
    int bad = 0, unstable = 0, my_masked = 0;
    double hsum = 0.0;
    for (int p = tid; p < L; p += blockDim.x) {
        const long long r = rowbase + p;
        const long long ifirst = r * a.nvec_row;
        const long long ilast = ifirst + a.nvec_row - 1;
        const int c0 = cta_of(ifirst, a.N, a.G);
        const int c1 = cta_of(ilast, a.N, a.G);
        RowState st{kEmptyMax, 0.0f, 0.0f, 0x7FFFFFFF, -INFINITY, -1};
        for (int cc = c0; cc <= c1; ++cc) {
            if (range_start(cc, a.N, a.G) >= range_start(cc + 1, a.N, a.G)) continue;
            const Partial q = a.partials[r + cc];
            merge_state(st, q.xm, q.S, q.T2, q.ai, q.best, q.bi, a.c);
        }
        float H = kLn2 * (log2f(st.S) - st.T2 / st.S);
        if (H < 0.0f) H = 0.0f;            // rounding below zero (NaN passes through)
        H = H + 0.0f;                      // -0 -> +0 so the key bits sort correctly
        bad |= (!isfinite(H) || !isfinite(st.xm)) ? 1 : 0;
        const bool masked = a.mask[r] != 0;
        my_masked += masked ? 1 : 0;
        const int A = st.ai;
        const int Y = masked ? st.bi : -1;
        Hs[p] = H;
        As[p] = A;
        Ys[p] = Y;
        a.entropy[r] = H;
        a.argmax[r] = A;
        a.sampled[r] = Y;
        a.selected[r] = 0;
        hsum += (double)H;
        unstable |= (a.prev_argmax[r] != A) ? 1 : 0;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            a.status[b] = EB_STATUS_NONFINITE;
            if (a.steps_taken) a.steps_taken[b] = a.step + 1;
            if (a.committed) a.committed[b] = 0;
            if (a.mean_entropy) a.mean_entropy[b] = NAN;
        }
        return;
    }
    if (my_masked) atomicAdd(&counts[1], my_masked);
    const double mean = block_sum_double(hsum, red) / (double)L;   // has barriers
    const bool stable = __syncthreads_or(unstable) == 0;
    const bool stop = a.step >= 1 && stable && mean < (double)a.stop_entropy;
    const int nm = counts[1];

    int my_commit = 0;
    int new_status = EB_RUNNING;
    if (stop) {
        // adaptive stop: every still-masked position takes its argmax
        for (int p = tid; p < L; p += blockDim.x) {
            const long long r = rowbase + p;
            if (a.mask[r]) {
                a.tokens[r] = As[p];
                a.mask[r] = 0;
                a.selected[r] = 1;
                ++my_commit;
            }
        }
        new_status = EB_STOP_ADAPTIVE;
    } else {
        // 2. bitonic sort of (H bits << 32 | p) for masked p; unmasked keys sort last
        int n2 = 1;
        while (n2 < L) n2 <<= 1;
        for (int i = tid; i < n2; i += blockDim.x) {
            unsigned long long k = ~0ull;
            if (i < L && a.mask[rowbase + i])
                k = ((unsigned long long)__float_as_uint(Hs[i]) << 32) | (unsigned)i;
            keys[i] = k;
        }
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < n2; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const unsigned long long x = keys[i], y = keys[ixj];
                        const bool asc = (i & k) == 0;
                        if ((x > y) == asc) {
                            keys[i] = y;
                            keys[ixj] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        // 3. inclusive prefix sums of the sorted entropies in binary64 (Hillis-Steele)
        for (int i = tid; i < n2; i += blockDim.x)
            scan[i] = (i < nm) ? (double)__uint_as_float((unsigned)(keys[i] >> 32)) : 0.0;
        __syncthreads();
        for (int off = 1; off < n2; off <<= 1) {
            double add[kMaxL / kK2Threads];
            int q = 0;
            for (int i = tid; i < n2; i += blockDim.x, ++q) add[q] = (i >= off) ? scan[i - off] : 0.0;
            __syncthreads();
            q = 0;
            for (int i = tid; i < n2; i += blockDim.x, ++q) scan[i] += add[q];
            __syncthreads();
        }
        // 4. accept sorted index i iff i == 0 or sum_{j<i} H_(j) <= bound; commit Y
        int my_left = 0;
        for (int i = tid; i < nm; i += blockDim.x) {
            const double before = (i == 0) ? 0.0 : scan[i - 1];
            const int pos = (int)(keys[i] & 0xFFFFFFFFu);
            const long long r = rowbase + pos;
            if (i == 0 || before <= (double)a.bound) {
                a.tokens[r] = Ys[pos];
                a.mask[r] = 0;
                a.selected[r] = 1;
                ++my_commit;
            } else {
                ++my_left;
            }
        }
        const bool any_left = __syncthreads_or(my_left) != 0;
        if (!any_left) {
            new_status = EB_STOP_COMPLETE;
        } else if (a.step >= a.max_steps - 1) {
            // step cap: the rest take their argmax (mask writes above are visible: barrier)
            for (int p = tid; p < L; p += blockDim.x) {
                const long long r = rowbase + p;
                if (a.mask[r]) {
                    a.tokens[r] = As[p];
                    a.mask[r] = 0;
                    a.selected[r] = 1;
                    ++my_commit;
                }
            }
            new_status = EB_STOP_CAP;
        }
    }
    for (int p = tid; p < L; p += blockDim.x) a.prev_argmax[rowbase + p] = As[p];
    if (my_commit) atomicAdd(&counts[0], my_commit);
    __syncthreads();
    if (tid == 0) {
        const int cnt = counts[0];
        if (new_status != EB_RUNNING) {
            a.status[b] = new_status;
            if (a.steps_taken) a.steps_taken[b] = a.step + 1;
        }
        if (a.committed) a.committed[b] = cnt;
        if (a.mean_entropy) a.mean_entropy[b] = (float)mean;
        if (a.committed_hist) a.committed_hist[(long long)b * a.max_steps + a.step] = cnt;
        if (a.mean_hist) a.mean_hist[(long long)b * a.max_steps + a.step] = (float)mean;
    }
}

}  // namespace ebk

// ====================================================================== host side

namespace {

thread_local std::string g_last_error;
// One-shot CUDA events recorded around the next row-statistics launch on this thread.
thread_local cudaEvent_t g_profile_begin = nullptr, g_profile_end = nullptr;

eb_status fail(eb_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

eb_status ok()
{
    g_last_error.clear();
    return EB_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Per-device launch geometry of the row-statistics kernels, filled once per device.
struct DeviceGeometry {
    std::atomic<int> ready{0};
    int grid[4] = {0, 0, 0, 0};   // SMs x resident CTAs for each element kind
};
DeviceGeometry g_geometry[64];

template <int KIND>
int resident_grid(int nsm)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ebk::k1_rowstats<KIND>,
                                                      ebk::kK1Threads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    long long g = (long long)nsm * per_sm;
    return (int)(g > ebk::kMaxGrid ? ebk::kMaxGrid : g);
}

eb_status geometry(int *grid_out, int kind)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(EB_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 64) return fail(EB_ERR_UNSUPPORTED, "device index %d >= 64", dev);
    DeviceGeometry &g = g_geometry[dev];
    if (g.ready.load(std::memory_order_acquire) == 0) {
        int nsm = 0;
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(EB_ERR_CUDA, "cudaDeviceGetAttribute failed");
        int grid[4] = {resident_grid<ebk::kF32Vec>(nsm), resident_grid<ebk::kBF16Vec>(nsm),
                       resident_grid<ebk::kF32Scalar>(nsm), resident_grid<ebk::kBF16Scalar>(nsm)};
        for (int i = 0; i < 4; ++i) g.grid[i] = grid[i];
        g.ready.store(1, std::memory_order_release);
    }
    *grid_out = g.grid[kind];
    return EB_OK;
}

ebk::RoundKeys round_keys(uint64_t seed)
{
    ebk::RoundKeys K;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        K.k[2 * r] = k0;
        K.k[2 * r + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return K;
}

float schedule_temperature(const eb_params *p, int step)
{
    if (p->max_steps <= 1) return p->t_start;
    return p->t_start + (p->t_end - p->t_start) * (float)step / (float)(p->max_steps - 1);
}

size_t partial_bytes(long long rows)
{
    return align256((size_t)(rows + ebk::kMaxGrid) * sizeof(ebk::Partial));
}

struct StepBuffers {
    uint8_t *mask;
    int32_t *tokens, *prev_argmax, *status, *steps_taken;
    float *entropy;
    int32_t *argmax, *sampled;
    uint8_t *selected;
    int32_t *committed;
    float *mean_entropy;
    int32_t *committed_hist;
    float *mean_hist;
};

eb_status check_common(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                       const void *d_logits, const StepBuffers &sb, void *d_ws, size_t ws_bytes)
{
    if (!params) return fail(EB_ERR_INVALID, "params is NULL");
    if (params->flags != 0) return fail(EB_ERR_INVALID, "params->flags must be 0");
    if (params->max_steps < 1) return fail(EB_ERR_INVALID, "max_steps must be >= 1");
    if (!(params->t_start > 0.0f) || !(params->t_end > 0.0f) || !std::isfinite(params->t_start) ||
        !std::isfinite(params->t_end))
        return fail(EB_ERR_INVALID, "temperatures must be finite and > 0");
    if (!std::isfinite(params->entropy_bound) || !std::isfinite(params->stop_entropy))
        return fail(EB_ERR_INVALID, "entropy_bound / stop_entropy must be finite");
    if (B < 0) return fail(EB_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (L < 1 || L > ebk::kMaxL) return fail(EB_ERR_INVALID, "L must be in [1, %d] (got %d)", ebk::kMaxL, L);
    if (V < 1) return fail(EB_ERR_INVALID, "V must be >= 1 (got %d)", V);
    if (dtype != EB_F32 && dtype != EB_BF16) return fail(EB_ERR_INVALID, "unknown dtype %d", (int)dtype);
    if (B == 0) return EB_OK;
    if (!d_logits) return fail(EB_ERR_INVALID, "d_logits is NULL");
    if (!sb.mask || !sb.tokens || !sb.prev_argmax || !sb.status || !sb.entropy || !sb.argmax ||
        !sb.sampled || !sb.selected)
        return fail(EB_ERR_INVALID, "a required state / output pointer is NULL");
    const long long rows = (long long)B * L;
    if (rows > (1ll << 31) - ebk::kMaxGrid) return fail(EB_ERR_UNSUPPORTED, "B*L too large");
    if (!d_ws) return fail(EB_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)d_ws & 255) != 0) return fail(EB_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < eb_workspace_bytes(B, L, V, dtype))
        return fail(EB_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes,
                    eb_workspace_bytes(B, L, V, dtype));
    return EB_OK;
}

// Enqueues k1 + k2 for one step.  Arguments were validated by the caller.
eb_status launch_step(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                      const void *d_logits, int step, float T, const StepBuffers &sb,
                      void *d_ws, cudaStream_t stream)
{
    const size_t esize = dtype == EB_F32 ? 4 : 2;
    const bool aligned = (((uintptr_t)d_logits & 15) == 0) && (((size_t)V * esize) % 16 == 0);
    int kind;
    if (dtype == EB_F32) kind = aligned ? ebk::kF32Vec : ebk::kF32Scalar;
    else kind = aligned ? ebk::kBF16Vec : ebk::kBF16Scalar;
    const int vec = kind == ebk::kF32Vec ? 4 : (kind == ebk::kBF16Vec ? 8 : 1);
    int gmax = 0;
    eb_status st = geometry(&gmax, kind);
    if (st != EB_OK) return st;
    const long long rows = (long long)B * L;
    const long long nvec_row = V / vec;
    const long long N = rows * nvec_row;
    if (N > (1ll << 48)) return fail(EB_ERR_UNSUPPORTED, "B*L*V too large");
    const int G = (int)(N < gmax ? N : gmax);

    ebk::K1Args a1;
    a1.logits = d_logits;
    a1.mask = sb.mask;
    a1.status = sb.status;
    a1.partials = static_cast<ebk::Partial *>(d_ws);
    a1.nvec_row = nvec_row;
    a1.N = N;
    a1.L = L;
    a1.G = G;
    a1.step = step;
    a1.c = ebk::kLog2e / T;
    a1.invT = 1.0f / T;
    a1.keys = round_keys(params->seed);
    cudaEvent_t prof_begin = g_profile_begin, prof_end = g_profile_end;
    g_profile_begin = g_profile_end = nullptr;
    if (prof_begin && cudaEventRecord(prof_begin, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");
    switch (kind) {
    case ebk::kF32Vec: ebk::k1_rowstats<ebk::kF32Vec><<<G, ebk::kK1Threads, 0, stream>>>(a1); break;
    case ebk::kBF16Vec: ebk::k1_rowstats<ebk::kBF16Vec><<<G, ebk::kK1Threads, 0, stream>>>(a1); break;
    case ebk::kF32Scalar: ebk::k1_rowstats<ebk::kF32Scalar><<<G, ebk::kK1Threads, 0, stream>>>(a1); break;
    default: ebk::k1_rowstats<ebk::kBF16Scalar><<<G, ebk::kK1Threads, 0, stream>>>(a1); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "row-statistics launch: %s", cudaGetErrorString(e));
    if (prof_end && cudaEventRecord(prof_end, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");

    ebk::K2Args a2;
    a2.partials = static_cast<const ebk::Partial *>(d_ws);
    a2.mask = sb.mask;
    a2.tokens = sb.tokens;
    a2.prev_argmax = sb.prev_argmax;
    a2.status = sb.status;
    a2.steps_taken = sb.steps_taken;
    a2.entropy = sb.entropy;
    a2.argmax = sb.argmax;
    a2.sampled = sb.sampled;
    a2.selected = sb.selected;
    a2.committed = sb.committed;
    a2.mean_entropy = sb.mean_entropy;
    a2.committed_hist = sb.committed_hist;
    a2.mean_hist = sb.mean_hist;
    a2.nvec_row = nvec_row;
    a2.N = N;
    a2.L = L;
    a2.G = G;
    a2.step = step;
    a2.max_steps = params->max_steps;
    a2.c = a1.c;
    a2.bound = params->entropy_bound;
    a2.stop_entropy = params->stop_entropy;
    ebk::k2_select<<<B, ebk::kK2Threads, 0, stream>>>(a2);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "selection launch: %s", cudaGetErrorString(e));
    return EB_OK;
}

}  // namespace

extern "C" {

eb_status eb_default_params(eb_params *p)
{
    if (!p) return fail(EB_ERR_INVALID, "params is NULL");
    p->max_steps = 48;
    p->t_start = 0.8f;
    p->t_end = 0.4f;
    p->entropy_bound = 0.1f;
    p->stop_entropy = 0.005f;
    p->flags = 0;
    p->seed = 0;
    return ok();
}

float eb_temperature(const eb_params *p, int step)
{
    if (!p) return 0.0f;
    return schedule_temperature(p, step);
}

size_t eb_workspace_bytes(int B, int L, int V, eb_dtype dtype)
{
    (void)V;
    (void)dtype;
    if (B < 0 || L < 1) return 0;
    return partial_bytes((long long)B * L);
}

eb_status eb_sampler_step(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                          const void *d_logits, int step, float temperature,
                          uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                          int32_t *d_status, int32_t *d_steps_taken,
                          float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                          uint8_t *d_selected, int32_t *d_committed, float *d_mean_entropy,
                          void *d_workspace, size_t workspace_bytes, void *stream)
{
    StepBuffers sb{d_mask, d_tokens, d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax,
                   d_sampled, d_selected, d_committed, d_mean_entropy, nullptr, nullptr};
    eb_status st = check_common(params, B, L, V, dtype, d_logits, sb, d_workspace, workspace_bytes);
    if (st != EB_OK) return st;
    if (B == 0) return ok();
    if (step < 0 || step >= params->max_steps)
        return fail(EB_ERR_INVALID, "step %d outside [0, max_steps=%d)", step, params->max_steps);
    if (std::isnan(temperature) || std::isinf(temperature))
        return fail(EB_ERR_INVALID, "temperature must be finite");
    const float T = temperature > 0.0f ? temperature : schedule_temperature(params, step);
    st = launch_step(params, B, L, V, dtype, d_logits, step, T, sb, d_workspace,
                     static_cast<cudaStream_t>(stream));
    return st == EB_OK ? ok() : st;
}

eb_status eb_sample_canvas(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                           eb_logits_fn logits_fn, void *user, void *d_logits, int start_step,
                           uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                           int32_t *d_status, int32_t *d_steps_taken,
                           int32_t *d_committed_per_step, float *d_mean_entropy_per_step,
                           float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                           uint8_t *d_selected, void *d_workspace, size_t workspace_bytes,
                           int poll_every, int *steps_run, void *stream)
{
    if (steps_run) *steps_run = 0;
    StepBuffers sb{d_mask, d_tokens, d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax,
                   d_sampled, d_selected, nullptr, nullptr, d_committed_per_step,
                   d_mean_entropy_per_step};
    eb_status st = check_common(params, B, L, V, dtype, d_logits, sb, d_workspace, workspace_bytes);
    if (st != EB_OK) return st;
    if (!logits_fn) return fail(EB_ERR_INVALID, "logits_fn is NULL");
    if (start_step < 0) return fail(EB_ERR_INVALID, "start_step must be >= 0");
    if (poll_every < 0) return fail(EB_ERR_INVALID, "poll_every must be >= 0");
    if (B == 0) return ok();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int ran = 0;
    for (int step = start_step; step < params->max_steps; ++step) {
        if (logits_fn(user, step, d_tokens, d_status, d_logits, stream) != 0) {
            if (steps_run) *steps_run = ran;
            return fail(EB_ERR_CALLBACK, "logits callback failed at step %d", step);
        }
        st = launch_step(params, B, L, V, dtype, d_logits, step, schedule_temperature(params, step),
                         sb, d_workspace, s);
        if (st != EB_OK) {
            if (steps_run) *steps_run = ran;
            return st;
        }
        ++ran;
        if (poll_every > 0 && (ran % poll_every) == 0 && step + 1 < params->max_steps) {
            // stop early once no canvas runs: read the status words back in small chunks
            bool any_running = false;
            int32_t chunk[256];
            for (int b0 = 0; b0 < B && !any_running; b0 += 256) {
                const int n = (B - b0) < 256 ? (B - b0) : 256;
                cudaError_t e = cudaMemcpyAsync(chunk, d_status + b0, n * sizeof(int32_t),
                                                cudaMemcpyDeviceToHost, s);
                if (e == cudaSuccess) e = cudaStreamSynchronize(s);
                if (e != cudaSuccess) {
                    if (steps_run) *steps_run = ran;
                    return fail(EB_ERR_CUDA, "status read-back: %s", cudaGetErrorString(e));
                }
                for (int i = 0; i < n; ++i) any_running |= (chunk[i] == EB_RUNNING);
            }
            if (!any_running) break;
        }
    }
    if (steps_run) *steps_run = ran;
    return ok();
}

const char *eb_status_string(eb_status s)
{
    switch (s) {
    case EB_OK: return "ok";
    case EB_ERR_INVALID: return "invalid argument";
    case EB_ERR_CUDA: return "CUDA error";
    case EB_ERR_UNSUPPORTED: return "unsupported";
    case EB_ERR_WORKSPACE: return "workspace too small or misaligned";
    case EB_ERR_CALLBACK: return "logits callback failed";
    }
    return "unknown status";
}

const char *eb_last_error(void) { return g_last_error.c_str(); }

eb_status eb_set_profile_events(void *k1_begin, void *k1_end)
{
    if ((k1_begin == nullptr) != (k1_end == nullptr))
        return fail(EB_ERR_INVALID, "give both profile events or neither");
    g_profile_begin = static_cast<cudaEvent_t>(k1_begin);
    g_profile_end = static_cast<cudaEvent_t>(k1_end);
    return ok();
}

}  // extern "C"
