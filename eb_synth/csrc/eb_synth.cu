// eb_synth.cu -- device side of the seeded synthetic-input generator (stand-in denoiser
// logits and fused-unembedding inputs).  Bit-identical to the numpy generator of the
// eb_synth package: every binary32 operation below is an explicitly rounded intrinsic
// (__fadd_rn / __fmul_rn / __fdiv_rn / __fsqrt_rn), so nothing is contracted into an FMA.
#include <cuda_runtime.h>

#include <cstdint>

#include "eb_synth.h"

namespace {

constexpr uint32_t kStreamNormal = 2u, kStreamPosition = 3u;
constexpr uint32_t kStreamUnembedH = 5u, kStreamUnembedCol = 6u, kStreamUnembedW = 7u;

__device__ __forceinline__ float bits(uint32_t b) { return __uint_as_float(b); }

// Philox4x32-10 (Salmon et al., SC'11).
__device__ __forceinline__ uint4 philox(uint4 c, uint64_t seed)
{
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1,
                       (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
    }
    return c;
}

__device__ __forceinline__ float uniform(uint32_t w)
{
    return __fmul_rn(__fadd_rn((float)(w >> 9), 0.5f), 1.1920928955078125e-07f);
}

// ln x for x in (0, 1): x = 2^e f, f in [sqrt(1/2), sqrt(2)), ln f = 2 atanh(s), s =
// (f-1)/(f+1), series through s^9; ln x = e ln2_hi + (e ln2_lo + ln f).
__device__ __forceinline__ float ln_f32(float x)
{
    const uint32_t xb = __float_as_uint(x);
    int e = (int)((xb >> 23) & 0xFFu) - 127;
    float f = bits((xb & 0x7FFFFFu) | 0x3F800000u);
    if (f > bits(0x3FB504F3u)) {
        f = __fmul_rn(f, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fadd_rn(f, -1.0f), __fadd_rn(f, 1.0f));
    const float z = __fmul_rn(s, s);
    float t = __fmul_rn(bits(0x3DE38E39u), z);
    t = __fadd_rn(t, bits(0x3E124925u));
    t = __fmul_rn(t, z);
    t = __fadd_rn(t, bits(0x3E4CCCCDu));
    t = __fmul_rn(t, z);
    t = __fadd_rn(t, bits(0x3EAAAAABu));
    const float a = __fadd_rn(s, s);
    const float lnf = __fadd_rn(a, __fmul_rn(a, __fmul_rn(z, t)));
    const float ef = (float)e;
    return __fadd_rn(__fmul_rn(ef, bits(0x3F317200u)), __fadd_rn(__fmul_rn(ef, bits(0x35BFBE8Eu)), lnf));
}

// (cos, sin)(2 pi u), u in (0, 1): octant reduction, Taylor series on [0, pi/4].
__device__ __forceinline__ void sincos_2pi(float u, float &cosv, float &sinv)
{
    const float t = __fmul_rn(u, 8.0f);
    const int o = (int)t;
    const float f = __fadd_rn(t, -(float)o);
    const float phi = (o & 1) ? __fadd_rn(1.0f, -f) : f;
    const float a = __fmul_rn(phi, bits(0x3F490FDBu));
    const float a2 = __fmul_rn(a, a);
    float q = __fmul_rn(bits(0x3638EF1Du), a2);
    q = __fadd_rn(q, bits(0xB9500D01u));
    q = __fmul_rn(q, a2);
    q = __fadd_rn(q, bits(0x3C088889u));
    q = __fmul_rn(q, a2);
    q = __fadd_rn(q, bits(0xBE2AAAABu));
    q = __fmul_rn(q, a2);
    const float sn = __fadd_rn(a, __fmul_rn(a, q));
    float c = __fmul_rn(bits(0xB493F27Eu), a2);
    c = __fadd_rn(c, bits(0x37D00D01u));
    c = __fmul_rn(c, a2);
    c = __fadd_rn(c, bits(0xBAB60B61u));
    c = __fmul_rn(c, a2);
    c = __fadd_rn(c, bits(0x3D2AAAABu));
    c = __fmul_rn(c, a2);
    c = __fadd_rn(c, bits(0xBF000000u));
    c = __fmul_rn(c, a2);
    const float cs = __fadd_rn(1.0f, c);
    const bool swap = (o == 1) || (o == 2) || (o == 5) || (o == 6);
    const float cm = swap ? sn : cs;
    const float sm = swap ? cs : sn;
    cosv = (o >= 2 && o <= 5) ? -cm : cm;
    sinv = (o >= 4) ? -sm : sm;
}

__device__ __forceinline__ void normals4(uint4 w, float (&n)[4])
{
    const float r0 = __fsqrt_rn(__fmul_rn(ln_f32(uniform(w.x)), -2.0f));
    const float r1 = __fsqrt_rn(__fmul_rn(ln_f32(uniform(w.z)), -2.0f));
    float c0, s0, c1, s1;
    sincos_2pi(uniform(w.y), c0, s0);
    sincos_2pi(uniform(w.w), c1, s1);
    n[0] = __fmul_rn(r0, c0);
    n[1] = __fmul_rn(r0, s0);
    n[2] = __fmul_rn(r1, c1);
    n[3] = __fmul_rn(r1, s1);
}

__device__ __forceinline__ uint16_t to_bf16(float x)
{
    const uint32_t b = __float_as_uint(x);
    return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

// Binary32 to OCP FP8 e4m3: nearest, ties to even; magnitudes above 448 (the largest finite
// value) saturate to it; NaN becomes 0x7F.  The same steps as the numpy generator's: the
// exponent e = floor(log2 |x|) (at least -6, the subnormal grid), q = rint(|x| 2^(3 - e)) in
// 0..16, a carry of q = 16 into the exponent, then code (e + 7) 8 + q - 8 (q >= 8) or q.
__device__ __forceinline__ uint32_t to_e4m3(float x)
{
    const uint32_t bits = __float_as_uint(x);
    if (isnan(x)) return 0x7Fu;
    const uint32_t sign = (bits >> 24) & 0x80u;
    const float a = fabsf(x);
    if (a > 448.0f) return sign | 0x7Eu;
    int e = (int)((bits >> 23) & 0xFFu) - 127;
    if (e < -6) e = -6;
    const float scale = __int_as_float((127 + 3 - e) << 23);     // 2^(3 - e), exact
    int q = (int)rintf(__fmul_rn(a, scale));
    if (q >= 16) {
        e += 1;
        q >>= 1;
    }
    const uint32_t code = q >= 8 ? (uint32_t)((e + 7) * 8 + (q - 8)) : (uint32_t)q;
    return sign | code;
}

constexpr int kThreads = 256;
constexpr int kGroupsPerThread = 8;

// grid: x = chunks of kThreads * kGroupsPerThread groups of 4 entries, y = row (b * L + p).
// With slot_block, output canvas b is a slot that holds canvas slot_block[b] of the recipe
// (skipped when negative) at step slot_step[b]; otherwise canvas b at `step`.
__global__ void __launch_bounds__(kThreads) peaked_logits_kernel(const eb_synth_recipe r, int step,
                                                                 const int32_t *status,
                                                                 const int32_t *slot_block,
                                                                 const int32_t *slot_step, void *out)
{
    __shared__ long long t_p;
    __shared__ float h_p;
    const long long row = blockIdx.y;
    const int ob = (int)(row / r.L);
    const uint32_t p = (uint32_t)(row - (long long)ob * r.L);
    int b = ob;
    if (slot_block) {
        b = slot_block[ob];
        if (b < 0 || b >= r.B) return;
        step = slot_step[ob];
    } else if (status && status[b] != 0) {
        return;
    }
    const uint64_t seed = r.seed[b];
    if (threadIdx.x == 0) {
        const uint4 w = philox(make_uint4(0u, p, 0u, (kStreamPosition << 24) | (uint32_t)b), seed);
        t_p = (long long)(((uint64_t)w.x * (uint64_t)(uint32_t)r.V) >> 32);
        float h = __fmul_rn(r.base_scale, uniform(w.y));
        h = __fadd_rn(h, r.base_lo);
        h_p = __fadd_rn(h, __fmul_rn(r.growth[b], (float)step));
    }
    __syncthreads();
    const long long nk = ((long long)r.V + 3) / 4;
    const uint32_t sw = (kStreamNormal << 24) | (uint32_t)b;
    const bool vec = (r.V % 4) == 0;
    for (int g = 0; g < kGroupsPerThread; ++g) {
        const long long k = ((long long)blockIdx.x * kGroupsPerThread + g) * kThreads + threadIdx.x;
        if (k >= nk) break;
        const uint4 w = philox(make_uint4((uint32_t)k, p, (uint32_t)step, sw), seed);
        float n[4];
        normals4(w, n);
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[j] = __fmul_rn(n[j], r.sigma);
            if (4 * k + j == t_p) x[j] = __fadd_rn(x[j], h_p);
        }
        const long long base = row * r.V + 4 * k;
        if (r.dtype == 0) {
            float *o = static_cast<float *>(out);
            if (vec) {
                *reinterpret_cast<float4 *>(o + base) = make_float4(x[0], x[1], x[2], x[3]);
            } else {
                for (int j = 0; j < 4; ++j)
                    if (4 * k + j < r.V) o[base + j] = x[j];
            }
        } else if (r.dtype == 1) {
            uint16_t *o = static_cast<uint16_t *>(out);
            if (vec) {
                const uint32_t lo = (uint32_t)to_bf16(x[0]) | ((uint32_t)to_bf16(x[1]) << 16);
                const uint32_t hi = (uint32_t)to_bf16(x[2]) | ((uint32_t)to_bf16(x[3]) << 16);
                *reinterpret_cast<uint2 *>(o + base) = make_uint2(lo, hi);
            } else {
                for (int j = 0; j < 4; ++j)
                    if (4 * k + j < r.V) o[base + j] = to_bf16(x[j]);
            }
        } else {
            uint8_t *o = static_cast<uint8_t *>(out);
            if (vec) {
                const uint32_t w = to_e4m3(x[0]) | (to_e4m3(x[1]) << 8) | (to_e4m3(x[2]) << 16) |
                                   (to_e4m3(x[3]) << 24);
                *reinterpret_cast<uint32_t *>(o + base) = w;
            } else {
                for (int j = 0; j < 4; ++j)
                    if (4 * k + j < r.V) o[base + j] = (uint8_t)to_e4m3(x[j]);
            }
        }
    }
}

// grid: x = chunks of groups, y = row; writes `cols` bf16 entries per row of N(0,1) * scale,
// plus `bias` at column col_of_row (computed from stream `col_stream` when >= 0).
__global__ void __launch_bounds__(kThreads) gaussian_bf16_kernel(uint64_t seed, uint32_t stream_id,
                                                                 int cols, float scale, float bias,
                                                                 int col_stream, uint16_t *out)
{
    __shared__ long long bias_col;
    const uint32_t rowi = blockIdx.y;
    if (threadIdx.x == 0) {
        bias_col = -1;
        if (col_stream >= 0) {
            const uint4 w = philox(make_uint4(0u, rowi, 0u, (uint32_t)col_stream << 24), seed);
            bias_col = (long long)(((uint64_t)w.x * (uint64_t)(uint32_t)cols) >> 32);
        }
    }
    __syncthreads();
    const long long nk = ((long long)cols + 3) / 4;
    for (int g = 0; g < kGroupsPerThread; ++g) {
        const long long k = ((long long)blockIdx.x * kGroupsPerThread + g) * kThreads + threadIdx.x;
        if (k >= nk) break;
        const uint4 w = philox(make_uint4((uint32_t)k, rowi, 0u, stream_id << 24), seed);
        float n[4];
        normals4(w, n);
        for (int j = 0; j < 4; ++j) {
            const long long v = 4 * k + j;
            if (v >= cols) break;
            float x = __fmul_rn(n[j], scale);
            if (v == bias_col) x = __fadd_rn(x, bias);
            out[(long long)rowi * cols + v] = to_bf16(x);
        }
    }
}

}  // namespace

extern "C" {

int eb_synth_logits(const eb_synth_recipe *r, int step, const int32_t *d_status, void *d_logits,
                    void *stream)
{
    if (!r || !d_logits || r->B < 0 || r->B > EB_SYNTH_MAX_B || r->L < 1 || r->V < 1 ||
        (r->dtype < 0 || r->dtype > 2) || step < 0 || (long long)r->B * r->L > 65535)
        return 1;
    if (r->B == 0) return 0;
    const long long nk = ((long long)r->V + 3) / 4;
    const long long per_cta = (long long)kThreads * kGroupsPerThread;
    dim3 grid((unsigned)((nk + per_cta - 1) / per_cta), (unsigned)(r->B * r->L));
    peaked_logits_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(*r, step, d_status,
                                                                                  nullptr, nullptr, d_logits);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

int eb_synth_slot_logits(const eb_synth_recipe *r, int B_slots, const int32_t *d_slot_block,
                         const int32_t *d_slot_step, void *d_logits, void *stream)
{
    if (!r || !d_logits || !d_slot_block || !d_slot_step || r->B < 1 || r->B > EB_SYNTH_MAX_B ||
        r->L < 1 || r->V < 1 || (r->dtype < 0 || r->dtype > 2) || B_slots < 0 ||
        (long long)B_slots * r->L > 65535)
        return 1;
    if (B_slots == 0) return 0;
    const long long nk = ((long long)r->V + 3) / 4;
    const long long per_cta = (long long)kThreads * kGroupsPerThread;
    dim3 grid((unsigned)((nk + per_cta - 1) / per_cta), (unsigned)(B_slots * r->L));
    peaked_logits_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(*r, 0, nullptr, d_slot_block,
                                                                                  d_slot_step, d_logits);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

int eb_synth_block_callback(void *user, int B, const int32_t *d_slot_block, const int32_t *d_slot_step,
                            const int32_t *d_tokens, void *d_logits, void *stream)
{
    (void)d_tokens;
    return eb_synth_slot_logits(static_cast<const eb_synth_recipe *>(user), B, d_slot_block, d_slot_step,
                                d_logits, stream);
}

int eb_synth_logits_callback(void *user, int step, const int32_t *d_tokens, const int32_t *d_status,
                             void *d_logits, void *stream)
{
    (void)d_tokens;
    return eb_synth_logits(static_cast<const eb_synth_recipe *>(user), step, d_status, d_logits,
                           stream);
}

int eb_synth_unembed_inputs(uint64_t seed, int M, int K, int V, float sigma_w, float bias,
                            uint16_t *d_h, uint16_t *d_W, void *stream)
{
    if (M < 1 || K < 1 || V < 1 || !d_h || !d_W || M > 65535 || K > 65535) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long per_cta = (long long)kThreads * kGroupsPerThread;
    dim3 gh((unsigned)((((long long)K + 3) / 4 + per_cta - 1) / per_cta), (unsigned)M);
    gaussian_bf16_kernel<<<gh, kThreads, 0, s>>>(seed, kStreamUnembedH, K, 1.0f, 0.0f, -1, d_h);
    dim3 gw((unsigned)((((long long)V + 3) / 4 + per_cta - 1) / per_cta), (unsigned)K);
    gaussian_bf16_kernel<<<gw, kThreads, 0, s>>>(seed, kStreamUnembedW, V, sigma_w, bias,
                                                 (int)kStreamUnembedCol, d_W);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
