// eb_sampler.cu -- kernels and C ABI of the B300 (sm_103a) Entropy-Bounded (EB) denoising
// sampler step of DiffusionGemma.  The algorithm and the kernel structure are described at
// the top of eb_kernels.cuh.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "eb_kernels.cuh"
#include "eb_sampler.h"

namespace ebk {

enum Kind { kF32Vec = 0, kBF16Vec = 1, kF32Scalar = 2, kBF16Scalar = 3, kFP8Vec = 4, kFP8Scalar = 5 };
constexpr int kKinds = 6;

// Logits per 16-byte vector of a vector kind.
template <int KIND> struct KindTraits;
template <> struct KindTraits<kF32Vec> { static constexpr int VEC = 4; };
template <> struct KindTraits<kBF16Vec> { static constexpr int VEC = 8; };
template <> struct KindTraits<kFP8Vec> { static constexpr int VEC = 16; };

// Philox words of the VEC entries of vector jvec (entries jvec*VEC ..).  The word of entry
// v is word v % 4 of counter (v / 4, p, s, stream << 24 | b).
template <int VEC>
__device__ __forceinline__ void gumbel_words(long long jvec, uint32_t p, uint32_t s, uint32_t sw,
                                             const RoundKeys &K, uint32_t (&w)[VEC])
{
    if constexpr (VEC == 8) {
        const uint4 u = philox((uint32_t)(2 * jvec), p, s, sw, K);
        const uint4 v = philox((uint32_t)(2 * jvec + 1), p, s, sw, K);
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        w[4] = v.x; w[5] = v.y; w[6] = v.z; w[7] = v.w;
    } else if constexpr (VEC == 4) {
        const uint4 u = philox((uint32_t)jvec, p, s, sw, K);
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else {
        const uint4 u = philox((uint32_t)(jvec >> 2), p, s, sw, K);
        const uint32_t q = (uint32_t)(jvec & 3);
        w[0] = q == 0 ? u.x : (q == 1 ? u.y : (q == 2 ? u.z : u.w));
    }
}

// The arithmetic values of a row of canvas b at position p: the launch's step and temperature,
// or the canvas's own when the launch carries per-canvas arrays (continuous batching), whose
// canvas id then also replaces b in the Philox counter.
__device__ __forceinline__ RowCtx row_ctx(const K1Args &a, int b, uint32_t p)
{
    RowCtx rc;
    if (a.canvas_step) {
        rc.c = a.canvas_c[b];
        rc.invT = a.canvas_invT[b];
        rc.step = (uint32_t)a.canvas_step[b];
        rc.sw = (kStreamGumbel << 24) | (uint32_t)a.canvas_id[b];
    } else {
        rc.c = a.c;
        rc.invT = a.invT;
        rc.step = (uint32_t)a.step;
        rc.sw = (kStreamGumbel << 24) | (uint32_t)b;
    }
    rc.p = p;
    return rc;
}

// One vector of VEC logits (entries jvec*VEC ..).  Every lane of the warp calls this with
// the same trip count; `valid` masks lanes without a vector.
template <int VEC, bool MASKED>
__device__ __forceinline__ void consume_vec(const float (&x)[VEC], bool valid, long long jvec,
                                            const K1Args &a, const RowCtx &rc,
                                            RowState &st, float &nb, float &K)
{
    float e[VEC];
    if (valid) {
        float vmax;
        if constexpr (VEC == 8) vmax = max3(max3(x[0], x[1], x[2]), max3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
        else if constexpr (VEC == 4) vmax = max3(x[0], x[1], fmaxf(x[2], x[3]));
        else vmax = x[0];
        if (vmax > st.xm) {
            // new running max: rescale the sums and take its first index as the argmax
            const float d = (st.xm - vmax) * rc.c;
            const float sc = ex2(d);
            st.T2 = sc == 0.0f ? 0.0f : sc * fmaf(d, st.S, st.T2);
            st.S = sc == 0.0f ? 0.0f : st.S * sc;
            int j0 = VEC - 1;
#pragma unroll
            for (int j = VEC - 1; j >= 0; --j)
                if (x[j] == vmax) j0 = j;
            st.ai = (int)(jvec * VEC + j0);
            st.xm = vmax;
            nb = -vmax * rc.c;
            if (MASKED) K = cand_scale(st.xm, st.best, rc.c);
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float t = fmaf(x[j], rc.c, nb);
            e[j] = ex2(t);
            st.S += e[j];
            st.T2 = fmaf(t, e[j], st.T2);
        }
    }
    if constexpr (MASKED) {
        uint32_t w[VEC];
        bool any = false;
        if (valid) {
            gumbel_words<VEC>(jvec, rc.p, rc.step, rc.sw, a.keys, w);
#pragma unroll
            for (int j = 0; j < VEC; ++j) any |= one_minus_u_plus(w[j]) < fmaf(e[j], K, kCandAdd);
        }
        if (__any_sync(0xFFFFFFFFu, any)) {
            if (any) {
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float f = one_minus_u_plus(w[j]);
                    if (f < fmaf(e[j], K, kCandAdd)) {
                        const float delta = f - kOneMinusHalfUlp;          // 1 - u, exact
                        const float E = -log1pf(-delta);                   // -ln u
                        const float score = x[j] * rc.invT - logf(E);
                        const int idx = (int)(jvec * VEC + j);
                        if (better(score, idx, st.best, st.bi)) {
                            st.best = score;
                            st.bi = idx;
                        }
                    }
                }
            }
            warp_best(st.best, st.bi);
            K = cand_scale(st.xm, st.best, rc.c);
        }
    }
}

// Builds the weight prefix P[0..rows] (and the per-row mask flags) in shared memory with
// all threads of the block.  Row weight: 0 for halted canvases, nvec * (masked ? w_m : w_u).
__device__ void build_prefix(const K1Args &a, uint32_t *P, uint8_t *mflag, uint32_t *scan)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    const int per = (a.rows + nth - 1) / nth;
    const int r0 = tid * per;
    uint32_t local = 0;
    for (int k = 0; k < per; ++k) {
        const int r = r0 + k;
        if (r >= a.rows) break;
        const uint8_t m = (!a.raw && a.mask[r]) ? 1 : 0;
        mflag[r] = m;
        const bool active = a.status[r / a.L] == EB_RUNNING;
        const uint32_t w = active ? (uint32_t)a.nvec_row * (uint32_t)(m ? kWeightMasked : kWeightUnmasked) : 0u;
        P[r] = w;
        local += w;
    }
    const int warp = tid >> 5, lane = tid & 31;
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        uint32_t run = 0;
        for (int w = 0; w < (nth + 31) / 32; ++w) {
            const uint32_t t = scan[w];
            scan[w] = run;
            run += t;
        }
        P[a.rows] = run;
    }
    __syncthreads();
    uint32_t base = scan[warp] + incl - local;
    for (int k = 0; k < per; ++k) {
        const int r = r0 + k;
        if (r >= a.rows) break;
        const uint32_t w = P[r];
        P[r] = base;
        base += w;
    }
    __syncthreads();
}

__device__ __forceinline__ void write_partial(Partial *dst, const RowState &s, int flags)
{
    Partial out;
    out.xm = s.xm;
    out.S = s.S;
    out.T2 = s.T2;
    out.ai = s.ai;
    out.best = s.best;
    out.bi = s.bi;
    out.flags = flags;
    out.pad = 0;
    *dst = out;
}

// Block reduction of the consumers' states and the partial write (consumer threads only).
// A NaN in any thread's sums is recorded before the merge can scale it away.
__device__ __forceinline__ void reduce_and_store(RowState st, const K1Args &a, float c, RowState *red,
                                                 uint32_t *redflag, int row, int flags)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool nan_here = __any_sync(0xFFFFFFFFu, isnan(st.S) || isnan(st.T2));
    warp_merge(st, c);
    if (lane == 0) {
        red[warp] = st;
        redflag[warp] = nan_here ? (uint32_t)kPartialNonfinite : 0u;
    }
    consumer_sync();
    if (warp == 0) {
        RowState s2 = lane < kConsumerWarps ? red[lane] : empty_state();
        const uint32_t nf = __reduce_or_sync(0xFFFFFFFFu, lane < kConsumerWarps ? redflag[lane] : 0u);
        warp_merge(s2, c);
        if (lane == 0 && EB_CHECK((long long)row + blockIdx.x < a.nslots, kCheckPartialSlot))
            write_partial(&a.partials[row + blockIdx.x], s2, flags | (int)nf);
    }
    consumer_sync();
}

// ------------------------------------------------------------------ streaming path
//
// Every warp is one unit of the weighted partition (its slot is row + global warp index) and
// streams its row segments: each lane stages its own 16-byte vectors in shared memory with
// cp.async, kAsyncDepth batches of U vectors ahead, so that no barrier is shared between
// lanes.  Warps merge their lanes with shuffles; no block barrier runs after the prefix is
// built.
constexpr int kDirectThreads = 512;
constexpr int kDirectWarps = kDirectThreads / 32;
constexpr int kDirectU = 2;             // vectors per lane per batch (binary32, bfloat16)
constexpr int kFP8U = 1;                // ... and for e4m3, whose vectors hold 16 logits
constexpr int kAsyncDepth = 4;          // batches in flight per lane
constexpr int kDirectStageBytes = kAsyncDepth * kDirectU * kDirectThreads * 16;

// L2 policy for the logits: evicted first, so that streaming them does not push out the
// workspace (partials, row units) that the selection kernel reads right after.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Plain 8-byte load (the e4m3 tail), bypassing L1, evict-first in L2.
__device__ __forceinline__ uint2 ld_stream8(const uint2 *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p), "l"(evict_first_policy()));
    return r;
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async16_at(uint32_t dst, const uint4 *src, uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}

// The same copy of src_size (16 or 0) bytes: the rest of the 16-byte slot is zero-filled, and
// with 0 nothing is read.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const uint4 *src, uint32_t src_size, uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
                 "r"(src_size), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr)
                 : "memory");
    return r;
}

// The nfull whole batches of a segment [j0, j1) starting at vector j0, and the staging of its
// ragged last batch (vectors jf = j0 + nfull kBatch .. j1, when jf < j1) behind them: its
// vectors at or past j1 are zero-filled without a read.  The ragged batch is left in the ring
// for the caller, at the returned ring offset, all copies complete.  The thread's staging slot
// for ring position d and vector u is at sbase + d kDepthStride + u kSlotStride; the ring
// offset and the global pointer advance by constants, so that no slot or address is
// recomputed from the batch index.  One copy of the batch body, so that the masked and
// unmasked loops of the SM's warps stay in the instruction cache together.
template <int VEC, int U, bool MASKED>
__device__ __forceinline__ uint32_t async_batches(const K1Args &a, const uint4 *src, uint32_t j0, uint32_t j1,
                                                  uint32_t nfull, const RowCtx &rc, const PhiloxRow &ph, f32x2 c2,
                                                  RowState &st, PackedSums &q, float &nb, f32x2 &nb2, float &K,
                                                  float &bt, uint32_t sbase)
{
    constexpr uint32_t kBatch = 32u * U;
    constexpr uint32_t kSlotStride = kDirectThreads * 16u;
    constexpr uint32_t kDepthStride = U * kSlotStride;
    constexpr uint32_t kRing = kAsyncDepth * kDepthStride;
    static_assert((kRing & (kRing - 1)) == 0, "the staging ring must be a power of two bytes");
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t pol = evict_first_policy();
    const uint4 *g = src + j0 + lane;
    // batch k of the segment into ring offset offk: whole batches plain, the ragged one
    // predicated vector by vector
    auto stage_batch = [&](uint32_t k, uint32_t offk) {
        if (k < nfull) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                cp_async16_at(sbase + offk + (uint32_t)u * kSlotStride, g + k * kBatch + 32u * (uint32_t)u, pol);
        } else if (j0 + k * kBatch < j1) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool in = j0 + k * kBatch + 32u * (uint32_t)u + lane < j1;
                cp_async16_zfill(sbase + offk + (uint32_t)u * kSlotStride, in ? g + k * kBatch + 32u * (uint32_t)u : src + j0,
                                 in ? 16u : 0u, pol);
            }
        }
    };
#pragma unroll
    for (int k = 0; k < kAsyncDepth - 1; ++k) {
        stage_batch((uint32_t)k, (uint32_t)k * kDepthStride);
        cp_async_commit();
    }
    uint32_t off = 0;                                        // ring offset of the batch consumed next
    uint32_t jv = j0 + lane;
#pragma unroll 1
    for (uint32_t b = 0; b < nfull; ++b) {
        // batch b + depth - 1, whole, ragged or past the end (nothing)
        stage_batch(b + (uint32_t)(kAsyncDepth - 1), (off + (uint32_t)(kAsyncDepth - 1) * kDepthStride) & (kRing - 1));
        cp_async_commit();
        cp_async_wait<kAsyncDepth - 1>();
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = lds128(sbase + off + (uint32_t)u * kSlotStride);
        consume_batch<VEC, U, MASKED>(r, jv, a, rc, ph, c2, st, q, nb, nb2, K, bt);
        off = (off + kDepthStride) & (kRing - 1);
        jv += kBatch;
    }
    cp_async_wait<0>();
    return off;
}

// One row segment [j0, j1) of a warp with a deep prefetch: each lane copies the vectors it
// will consume with cp.async (16 bytes each, L2 evict-first, no L1) into its own
// shared-memory slots, kAsyncDepth batches ahead, and waits only for its own oldest group (no
// cross-lane barrier).  Whole batches run in a masked or an unmasked instance of the loop.
// The ragged last batch is staged in the ring behind them and taken vector by vector (for
// e4m3, whose half vectors must stay in lane order, with plain guarded loads instead).
template <int VEC, int U>
__device__ __forceinline__ void async_segment(const K1Args &a, const uint4 *src, uint32_t j0, uint32_t j1,
                                              const RowCtx &rc, f32x2 c2, RowState &st, PackedSums &q,
                                              bool gumbel, uint4 *stage)
{
    constexpr uint32_t kBatch = 32u * U;
    constexpr uint32_t kSlotStride = kDirectThreads * 16u;
    const uint32_t lane = threadIdx.x & 31;
    float nb = -st.xm * rc.c;
    f32x2 nb2 = pk2(nb, nb);
    float K = cand_scale(st.xm, st.best, rc.c);
    const uint32_t nfull = (j1 - j0) / kBatch;
    const uint32_t jf = j0 + nfull * kBatch;
    const uint32_t sbase = smem_addr(stage) + threadIdx.x * 16u;
    const uint32_t js = VEC == 16 ? jf : j1;       // end of what goes through the ring
    float bt = -INFINITY;                  // the seed threshold (a lower bound of the best score)
    uint32_t off = 0;
    if (j0 < js) {
        if (gumbel) {
            const PhiloxRow ph = philox_row(rc.p, rc.step, rc.sw, a.keys);
            off = async_batches<VEC, U, true>(a, src, j0, js, nfull, rc, ph, c2, st, q, nb, nb2, K, bt, sbase);
        } else {
            off = async_batches<VEC, U, false>(a, src, j0, js, nfull, rc, PhiloxRow{}, c2, st, q, nb, nb2, K, bt,
                                               sbase);
        }
    }
    if constexpr (VEC == 16) {
        // e4m3: the tail in half vectors of 8 logits, consecutive half vectors on consecutive
        // lanes, so that the lanes' entries stay in index order (first index on ties)
        const uint2 *src2 = reinterpret_cast<const uint2 *>(src);
#pragma unroll 1
        for (uint32_t hb = 2u * jf; hb < 2u * j1; hb += 32u) {
            const uint32_t h = hb + lane;
            const bool valid = h < 2u * j1;
            const uint2 r = valid ? ld_stream8(src2 + h) : make_uint2(0u, 0u);
            float x[8];
            e4m3x4_to_f32(r.x, x[0], x[1], x[2], x[3]);
            e4m3x4_to_f32(r.y, x[4], x[5], x[6], x[7]);
            consume_vals<8, true, true>(x, valid, h * 8u, a, rc, c2, st, q, nb, nb2, K, gumbel);
        }
    } else {
        // the ragged batch from the ring: its vector u of every lane, u = 0, 1, .. while any
        // lane's vector is inside the segment
#pragma unroll 1
        for (uint32_t u = 0; jf + 32u * u < j1; ++u) {
            const uint32_t idx = jf + 32u * u + lane;
            const bool valid = idx < j1;
            const uint4 r = valid ? lds128(sbase + off + u * kSlotStride) : make_uint4(0u, 0u, 0u, 0u);
            consume_packed<VEC, true>(r, valid, idx, a, rc, c2, st, q, nb, nb2, K, gumbel);
        }
    }
}

template <int KIND, int U>
__global__ void __launch_bounds__(kDirectThreads, 1) k1_rowstats_direct(const K1Args a)
{
    using Tr = KindTraits<KIND>;
    constexpr int VEC = Tr::VEC;
    __shared__ uint32_t P[kMaxWeightedRows + 1];
    __shared__ uint8_t mflag[kMaxWeightedRows];
    __shared__ uint32_t scan[32];
    extern __shared__ __align__(16) uint4 stage[];   // kAsyncDepth x U x kDirectThreads vectors
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the dependent selection grid may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    if (a.weighted) build_prefix(a, P, mflag, scan);
    __syncthreads();
    if (a.weighted && blockIdx.x == 0)
        for (int r = tid; r <= a.rows; r += blockDim.x) a.prefix_out[r] = P[r];
    // units are dealt round-robin over the CTAs, so every SM runs a mix of masked (ALU-heavy)
    // and unmasked (memory-heavy) row pieces rather than one kind
    const int gw = warp * gridDim.x + blockIdx.x;
    const Partition part{P, a.nvec_row, a.rows, a.weighted};
    SegmentCursor cur;
    cur.begin(part, gw, a.G);
    int row;
    long long j0, j1;
    while (cur.next(row, j0, j1)) {
        if (!EB_CHECK(row >= 0 && row < a.rows && j0 >= 0 && j0 <= j1 && j1 <= a.nvec_row, kCheckSegment)) continue;
        const int b = row / a.L;
        if (!a.weighted && a.status[b] != EB_RUNNING) continue;
        const RowCtx rc = row_ctx(a, b, (uint32_t)(row - b * a.L));
        const f32x2 c2 = pk2(rc.c, rc.c);
        const bool masked = !a.raw && (a.weighted ? mflag[row] != 0 : a.mask[row] != 0);
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.logits) +
                                                           (size_t)row * (size_t)a.row_bytes);
        RowState st = empty_state();
        PackedSums q;
        packed_zero(q);
        async_segment<VEC, U>(a, src, (uint32_t)j0, (uint32_t)j1, rc, c2, st, q, masked, stage);
        packed_fold(q, st);
        const bool nan_here = __any_sync(0xFFFFFFFFu, isnan(st.S) || isnan(st.T2));
        warp_merge(st, rc.c);
        if (lane == 0 && EB_CHECK((long long)row + gw < a.nslots, kCheckPartialSlot)) {
            write_partial(&a.partials[row + gw], st, nan_here ? kPartialNonfinite : 0);
            if (cur.first) a.rowunits[row].x = gw;
            if (cur.last) a.rowunits[row].y = gw;
        }
    }
}

// Scalar path (rows not 16-byte aligned): direct element loads, one entry per "vector".
template <int KIND>
__global__ void __launch_bounds__(kConsumers, 1) k1_rowstats_scalar(const K1Args a)
{
    __shared__ uint32_t P[kMaxWeightedRows + 1];
    __shared__ uint8_t mflag[kMaxWeightedRows];
    __shared__ RowState red[kConsumerWarps];
    __shared__ uint32_t scan[32];
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.launch_dependents;");
    if (a.weighted) build_prefix(a, P, mflag, scan);
    __syncthreads();
    if (a.weighted && blockIdx.x == 0)
        for (int r = tid; r <= a.rows; r += blockDim.x) a.prefix_out[r] = P[r];
    const Partition part{P, a.nvec_row, a.rows, a.weighted};
    SegmentCursor cur;
    cur.begin(part, blockIdx.x, a.G);
    int row;
    long long j0, j1;
    while (cur.next(row, j0, j1)) {
        if (!EB_CHECK(row >= 0 && row < a.rows && j0 >= 0 && j0 <= j1 && j1 <= a.nvec_row, kCheckSegment)) continue;
        const int b = row / a.L;
        if (!a.weighted && a.status[b] != EB_RUNNING) continue;
        const RowCtx rc = row_ctx(a, b, (uint32_t)(row - b * a.L));
        const bool masked = !a.raw && (a.weighted ? mflag[row] != 0 : a.mask[row] != 0);
        const char *base = static_cast<const char *>(a.logits) + (size_t)row * (size_t)a.row_bytes;
        RowState st = empty_state();
        float nb = -st.xm * rc.c;
        float K = cand_scale(st.xm, st.best, rc.c);
        for (long long j = j0; j < j1; j += kConsumers) {
            const long long v = j + tid;
            const bool valid = v < j1;
            float x[1] = {0.0f};
            if (valid) {
                if (KIND == kF32Scalar) x[0] = __ldg(reinterpret_cast<const float *>(base) + v);
                else if (KIND == kBF16Scalar)
                    x[0] = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(base) + v) << 16);
                else x[0] = e4m3_to_f32((uint32_t)__ldg(reinterpret_cast<const unsigned char *>(base) + v));
            }
            if (masked) consume_vec<1, true>(x, valid, v, a, rc, st, nb, K);
            else consume_vec<1, false>(x, valid, v, a, rc, st, nb, K);
        }
        reduce_and_store(st, a, rc.c, red, scan, row, 0);
        if (tid == 0) {
            if (cur.first) a.rowunits[row].x = blockIdx.x;
            if (cur.last) a.rowunits[row].y = blockIdx.x;
        }
    }
}

// ------------------------------------------------------------------ selection kernel

__device__ __forceinline__ unsigned long long k2_row_start(const K2Args &a, long long r)
{
    return a.weighted ? (unsigned long long)a.prefix[r]
                      : (unsigned long long)r * (unsigned long long)a.nvec_row;
}

constexpr int kSelGeneral = 4;  // selection flag: more than 32 low-entropy candidates (bits 0-1: halt)
constexpr int kMergeBatch = 6;   // partial states fetched per round by the selection kernel
// The selection kernel stages a canvas's partial states (one contiguous slot range on the
// streaming partition) in shared memory when the range holds at most this many slots.
constexpr int kK2StageSlots = 4096;
constexpr int kK2StageBytes = kK2StageSlots * (int)sizeof(Partial);

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
        v = o < v ? o : v;
    }
    return v;
}

__device__ __forceinline__ unsigned long long entropy_key(float H, int p)
{
    return ((unsigned long long)__float_as_uint(H) << 32) | (unsigned)p;
}

// One CTA per canvas.  Selection without a full sort: the positions with H <= bound
// (fixed point) come first in (H, p) order, so only they need sorting, followed by the
// lowest-entropy position above the bound, which is accepted iff every low one was and
// their sum stays within the bound.  No later position can be accepted.
// Merges the partial states of row r in slot order: the fused kernel's (group rank, column
// group) slots when k3_g > 0, else the streaming units u.x .. u.y of `rowunits`.  W and G: the
// streaming partition's total weight and unit count (a unit whose weight range is empty wrote
// nothing, only when W < G).
// `half` (0 or 1): this thread merges the first or the second half of the row's slots (the two
// threads of a row combine their halves in that order afterwards).
// `staged` (streaming partition only): the slots from staged_first on, copied to shared memory.
__device__ __forceinline__ void k2_merge_row(const K2Args &a, const Partial *partials, const int2 *rowunits,
                                             unsigned long long W, unsigned long long G, long long r, float c,
                                             int half, RowState &st, int &flags, const int2 *local_units = nullptr,
                                             int p = 0, const Partial *staged = nullptr, long long staged_first = 0)
{
    long long base, stride;
    int n;
    if (a.k3_g > 0) {
        const long long mb = r >> 7, rl = r & 127;
        base = mb * a.k3_g * a.k3_groups * 128 + rl;
        stride = 128;
        n = a.k3_groups * a.k3_g;
    } else {
        const int2 u = local_units ? local_units[p] : rowunits[r];
        base = r + u.x;
        stride = 1;
        n = u.y - u.x + 1;
        if (!EB_CHECK(u.x >= 0 && u.x <= u.y && (unsigned long long)u.y < G, kCheckUnits)) n = 0;
    }
    const int h = (n + 1) >> 1;
    const int lo = half ? h : 0, hi = half ? n : h;
    if (staged) {
        // from shared memory: a plain loop in slot order
#pragma unroll 1
        for (int i = lo; i < hi; ++i) {
            if (W < G) {
                const unsigned long long cu = (unsigned long long)(base - r + i);
                if (cu * W / G >= (cu + 1) * W / G) continue;
            }
            if (!EB_CHECK(base + i >= staged_first && base + i - staged_first < (long long)kK2StageSlots, kCheckPartialSlot))
                continue;
            const Partial q = staged[base + i - staged_first];
            merge_state(st, q.xm, q.S, q.T2, q.ai, q.best, q.bi, c);
            flags |= q.flags;
        }
        return;
    }
    // loads in batches of kMergeBatch independent requests, merged in slot order
    for (int i0 = lo; i0 < hi; i0 += kMergeBatch) {
        Partial q[kMergeBatch];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k)
            if (i0 + k < hi) {
                const long long slot = base + (long long)(i0 + k) * stride;
                if (EB_CHECK(slot >= 0 && slot < a.nslots, kCheckPartialSlot)) q[k] = partials[slot];
                else q[k] = Partial{-INFINITY, 0.0f, 0.0f, 0x7FFFFFFF, -INFINITY, -1, 0, 0};
            }
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            if (i0 + k >= hi) break;
            if (a.k3_g == 0 && W < G) {
                const unsigned long long cu = (unsigned long long)(base - r + i0 + k);
                if (cu * W / G >= (cu + 1) * W / G) continue;
            }
            merge_state(st, q[k].xm, q[k].S, q[k].T2, q[k].ai, q[k].best, q[k].bi, c);
            flags |= q[k].flags;
        }
    }
}

// The two threads of a row (lanes 2k, 2k + 1): the even one merges the odd one's state into
// its own, the even one's half of the slots first.
__device__ __forceinline__ void pair_combine(RowState &st, int &flags, float c)
{
    const float xm = __shfl_xor_sync(0xFFFFFFFFu, st.xm, 1);
    const float S = __shfl_xor_sync(0xFFFFFFFFu, st.S, 1);
    const float T2 = __shfl_xor_sync(0xFFFFFFFFu, st.T2, 1);
    const int ai = __shfl_xor_sync(0xFFFFFFFFu, st.ai, 1);
    const float best = __shfl_xor_sync(0xFFFFFFFFu, st.best, 1);
    const int bi = __shfl_xor_sync(0xFFFFFFFFu, st.bi, 1);
    const int of = __shfl_xor_sync(0xFFFFFFFFu, flags, 1);
    if ((threadIdx.x & 1) == 0) {
        merge_state(st, xm, S, T2, ai, best, bi, c);
        flags |= of;
    }
}

__global__ void __launch_bounds__(kK2Threads) k2_select(const K2Args a)
{
    __shared__ unsigned long long Hq[kMaxL];     // entropies in 2^-40 nats
    __shared__ float Hf[kMaxL];                  // entropies (binary32)
    __shared__ unsigned long long keys[kMaxL];   // low-entropy candidates
    __shared__ unsigned long long scanbuf[kMaxL];
    __shared__ int As[kMaxL];
    __shared__ int Ys[kMaxL];
    __shared__ uint8_t Ms[kMaxL];                // masked before this step
    __shared__ int Pv[kMaxL];                    // argmax of the previous step
    __shared__ uint8_t Acc[kMaxL];               // accepted at this step
    __shared__ unsigned long long red_sum[kK2Threads / 32];
    __shared__ unsigned long long red_min[kK2Threads / 32];
    __shared__ int4 red_cnt[kK2Threads / 32];   // per warp: masked, small, bad flags, unstable
    __shared__ uint32_t wtot[kK2Threads / 32];
    // per row: first and last partition unit (phase 1 only; shares the general sort's scan buffer)
    int2 *Ru = reinterpret_cast<int2 *>(scanbuf);
    __shared__ int n_gather, n_acc, sel_status, sel_committed, sel_flag, sel_stop, sel_ns, sel_nm, sel_cap;
    __shared__ float sel_mean;
    __shared__ unsigned long long sel_bigmin;
    extern __shared__ __align__(16) unsigned char k2_stage[];   // kK2StageBytes: staged partials

    const int b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = a.L;
    if (a.status[b] != EB_RUNNING) return;       // CTA-uniform
    // the canvas's own step and c under continuous batching, else the launch's
    const int step = a.canvas_step ? a.canvas_step[b] : a.step;
    const float cb = a.canvas_c ? a.canvas_c[b] : a.c;
    if (tid == 0) n_gather = 0;
    const long long rowbase = (long long)b * L;
    // launched as a programmatic dependent of the row-statistics kernel: the mask and the
    // previous argmax are not written by it, so they load while it drains; wait for its
    // partial states here
    for (int p = tid; p < L; p += blockDim.x) {
        Ms[p] = a.mask[rowbase + p] ? 1 : 0;
        Pv[p] = a.prev_argmax[rowbase + p];
    }
    // One canvas on the weighted partition: the row statistics' partition is a function of this
    // canvas's mask alone, so each row's first and last partition unit are computed here, before
    // the wait, instead of being read after it.  Unit g covers weight [g W / G, (g + 1) W / G),
    // so the unit holding weight position x is ((x + 1) G - 1) / W.
    const bool local = a.weighted && a.k3_g == 0 && a.rows == L && !a.canvas_step;
    unsigned long long Wloc = 0;
    if (local) {
        __syncthreads();                          // Ms complete
        const uint32_t wm = (uint32_t)a.nvec_row * (uint32_t)kWeightMasked;
        const uint32_t wu = (uint32_t)a.nvec_row * (uint32_t)kWeightUnmasked;
        // exclusive scan of the row weights, two rows per thread (L <= 1024 = 2 x 512)
        const int p0 = 2 * tid;
        const uint32_t w0 = p0 < L ? (Ms[p0] ? wm : wu) : 0u;
        const uint32_t w1 = p0 + 1 < L ? (Ms[p0 + 1] ? wm : wu) : 0u;
        const uint32_t mine = w0 + w1;
        uint32_t incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w = 0; w < kK2Threads / 32; ++w) {
            const uint32_t t = wtot[w];
            if (w < warp) before += t;
            total += t;
        }
        const unsigned long long Wt = total, Gt = (unsigned long long)a.G;
        const unsigned long long x0 = before + incl - mine;      // weight before row p0
        auto unit = [&](unsigned long long x) { return (int)(((x + 1ull) * Gt - 1ull) / Wt); };
        if (p0 < L) Ru[p0] = make_int2(unit(x0), unit(x0 + w0 - 1ull));
        if (p0 + 1 < L) Ru[p0 + 1] = make_int2(unit(x0 + w0), unit(x0 + w0 + w1 - 1ull));
        Wloc = Wt;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // On the streaming partition the canvas's partial states are one contiguous slot range, from
    // its first row's first unit to its last row's last unit: every thread copies its share of
    // it to shared memory at once (one round trip), and the rows merge from there.
    const Partial *staged = nullptr;
    long long staged_first = 0;
    if (a.k3_g == 0) {
        if (local) __syncthreads();               // Ru complete
        const int2 uf = local ? Ru[0] : a.rowunits[rowbase];
        const int2 ul = local ? Ru[L - 1] : a.rowunits[rowbase + L - 1];
        const long long s0 = rowbase + uf.x, s1 = rowbase + L - 1 + ul.y;
        if (s1 >= s0 && s1 - s0 < (long long)kK2StageSlots && EB_CHECK(s0 >= 0 && s1 < a.nslots, kCheckPartialSlot)) {
            Partial *pst = reinterpret_cast<Partial *>(k2_stage);
            const uint4 *src = reinterpret_cast<const uint4 *>(a.partials + s0);
            const uint32_t dst = smem_addr(pst);
            const int nchunk = (int)(s1 - s0 + 1) * (int)(sizeof(Partial) / 16);
            for (int i = tid; i < nchunk; i += blockDim.x)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16u * (uint32_t)i), "l"(src + i)
                             : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            staged = pst;
            staged_first = s0;
        }
    }
    const unsigned long long W = local ? Wloc : k2_row_start(a, a.rows);
    const unsigned long long G = (unsigned long long)a.G;
    const unsigned long long Wr = !a.raw_partials ? 0ull
                                  : a.raw_weighted ? (unsigned long long)a.raw_prefix[a.rows]
                                                   : (unsigned long long)a.rows * (unsigned long long)a.nvec_row;
    const unsigned long long Gr = (unsigned long long)a.raw_G;
    __syncthreads();

    // 1. merge each row's partials (ascending unit) -> H, A, Y.  Two threads per row: each merges
    // half of the row's slots, then the first half takes the second's state (a fixed order, so
    // the result does not depend on timing) and carries on alone.
    unsigned long long my_sum = 0, my_bigmin = ~0ull;
    int my_unstable = 0, my_bad = 0, my_masked = 0, my_small = 0;
    const int half = tid & 1;
    for (int p0 = 0; p0 < L; p0 += (int)(blockDim.x >> 1)) {
        const int p = p0 + (tid >> 1);
        const bool row_here = p < L;             // the same for both threads of a pair
        const long long r = rowbase + (row_here ? p : 0);
        RowState st = empty_state();
        int flags = 0;
        if (row_here)
            k2_merge_row(a, a.partials, a.rowunits, W, G, r, cb, half, st, flags, local ? Ru : nullptr, p, staged,
                         staged_first);
        pair_combine(st, flags, cb);
        RowState sr = empty_state();
        int rflags = 0;
        if (a.raw_partials) {
            // EB_FLAG_STOP_RAW_ENTROPY: the raw-logit (T = 1) pass's partial states, same scheme
            if (row_here) k2_merge_row(a, a.raw_partials, a.raw_rowunits, Wr, Gr, r, kLog2e, half, sr, rflags);
            pair_combine(sr, rflags, kLog2e);
        }
        if (!row_here || half) continue;
        float H = kLn2 * (log2f(st.S) - st.T2 / st.S);
        if (H < 0.0f) H = 0.0f;                  // rounding below zero (NaN passes through)
        H = H + 0.0f;                            // -0 -> +0 so the key bits order correctly
        if (!isfinite(H) || !isfinite(st.xm) || (flags & kPartialNonfinite)) my_bad |= 1;
        if (flags & kPartialTimeout) my_bad |= 2;
        const bool bad = my_bad != 0;
        const uint8_t m = Ms[p];
        const int A = st.ai;
        const int Y = m ? st.bi : -1;
        const unsigned long long hq = bad ? 0ull : (unsigned long long)__float2ull_rn(H * 1099511627776.0f);
        unsigned long long hstat = hq;           // the entropy the stop rule sums
        if (a.raw_partials) {
            // EB_FLAG_STOP_RAW_ENTROPY: the entropy of the raw logits (T = 1), same fixed point
            float Hr = kLn2 * (log2f(sr.S) - sr.T2 / sr.S);
            if (Hr < 0.0f) Hr = 0.0f;
            if (!isfinite(Hr) || (rflags & kPartialNonfinite)) my_bad |= 1;
            if (rflags & kPartialTimeout) my_bad |= 2;
            hstat = my_bad ? 0ull : (unsigned long long)__float2ull_rn(Hr * 1099511627776.0f);
        }
        Hq[p] = hq;
        Hf[p] = H;
        As[p] = A;
        Ys[p] = Y;
        Acc[p] = 0;
        a.entropy[r] = H;
        a.argmax[r] = A;
        a.sampled[r] = Y;
        // the stop statistics: every position, or the still-masked ones only
        if (m || !a.stop_masked_only) {
            my_sum += hstat;
            my_unstable |= (Pv[p] != A) ? 1 : 0;
        }
        if (m) {
            ++my_masked;
            if ((long long)hq <= a.bound_q) {
                ++my_small;
            } else {
                const unsigned long long key = entropy_key(H, p);
                my_bigmin = key < my_bigmin ? key : my_bigmin;
            }
        }
    }
    // the canvas statistics: warp reductions into one shared slot per warp and one barrier;
    // then warp 0 alone reduces the slots, takes the stop decision and, with at most 32
    // low-entropy candidates, the whole selection, while the other warps wait at the next barrier
    {
        const unsigned long long ws = warp_sum_u64(my_sum);
        const unsigned long long wm = warp_min_u64(my_bigmin);
        const int wcnt_m = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)my_masked);
        const int wcnt_s = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)my_small);
        const int wbad = (int)__reduce_or_sync(0xFFFFFFFFu, (unsigned)my_bad);
        const int wuns = (int)__reduce_or_sync(0xFFFFFFFFu, (unsigned)my_unstable);
        if (lane == 0) {
            red_sum[warp] = ws;
            red_min[warp] = wm;
            red_cnt[warp] = make_int4(wcnt_m, wcnt_s, wbad, wuns);
        }
    }
    __syncthreads();
    constexpr int kNW = kK2Threads / 32;
    if (warp == 0) {
        const unsigned long long sumq = warp_sum_u64(lane < kNW ? red_sum[lane] : 0ull);
        const unsigned long long bigmin = warp_min_u64(lane < kNW ? red_min[lane] : ~0ull);
        const int4 cw = lane < kNW ? red_cnt[lane] : make_int4(0, 0, 0, 0);
        const int nm = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)cw.x);
        const int ns = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)cw.y);
        const int badf = (int)__reduce_or_sync(0xFFFFFFFFu, (unsigned)cw.z);
        const bool stable = __reduce_or_sync(0xFFFFFFFFu, (unsigned)cw.w) == 0u;
        const int nstat = a.stop_masked_only ? nm : L;
        const long long stop_q =
            a.stop_masked_only ? (long long)ceil(a.stop_entropy * (double)nstat * 1099511627776.0) : a.stop_q;
        const bool stop = !badf && step >= 1 && stable && nstat > 0 && (long long)sumq < stop_q;
        const bool at_cap = step >= a.max_steps - 1;
        if (lane == 0) {
            sel_mean = nstat > 0 ? (float)sumq * 9.094947017729282e-13f / (float)nstat : NAN;   // 2^-40
            sel_flag = badf ? badf : 0;
            sel_stop = stop ? 1 : 0;
        }
        if (badf) {
            // nothing to select
        } else if (stop) {
            // adaptive stop: every still-masked position takes its argmax (in the commit pass)
            if (lane == 0) {
                sel_status = EB_STOP_ADAPTIVE;
                sel_committed = nm;
            }
        } else if (nm == 0) {
            if (lane == 0) {
                sel_status = EB_STOP_COMPLETE;
                sel_committed = 0;
            }
        } else if (ns <= 32) {
            // gather the low-entropy candidates in position order by ballot, sort them, accept
            // the prefix, then the lowest position above the bound if the prefix allows
            int cnt = 0;
            for (int p0 = 0; p0 < L; p0 += 32) {
                const int p = p0 + lane;
                const bool cand = p < L && Ms[p] && (long long)Hq[p] <= a.bound_q;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, cand);
                if (cand) keys[cnt + __popc(bal & ((1u << lane) - 1u))] = entropy_key(Hf[p], p);
                cnt += __popc(bal);
            }
            __syncwarp();
            unsigned long long k = lane < ns ? keys[lane] : ~0ull;
            // bitonic sort of 32 keys across the warp, ascending
#pragma unroll
            for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, k, stride);
                    const bool up = (lane & size) == 0;
                    const bool lower = (lane & stride) == 0;
                    const unsigned long long lo = o < k ? o : k, hi = o < k ? k : o;
                    k = (lower == up) ? lo : hi;
                }
            }
            const int pos = (int)(k & 0xFFFFFFFFu);
            const bool pos_ok = lane < ns && EB_CHECK(pos >= 0 && pos < L, kCheckRow);
            const unsigned long long h = pos_ok ? Hq[pos] : 0ull;
            unsigned long long incl = h;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                if (lane >= off) incl += o;
            }
            const unsigned long long excl = incl - h;
            const bool acc = lane < ns && (lane == 0 || (long long)excl <= a.bound_q);
            if (acc && pos_ok) Acc[pos] = 1;
            const unsigned acc_mask = __ballot_sync(0xFFFFFFFFu, acc);
            const unsigned ok_mask = __ballot_sync(0xFFFFFFFFu, acc || lane >= ns);
            const unsigned long long tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (lane == 0) {
                int nacc = __popc(acc_mask);
                // sorted index ns: the lowest-entropy position above the bound
                if (bigmin != ~0ull && (ns == 0 || (ok_mask == 0xFFFFFFFFu && (long long)tot <= a.bound_q))) {
                    const int bp = (int)(bigmin & 0xFFFFFFFFu);
                    if (EB_CHECK(bp >= 0 && bp < L, kCheckRow)) Acc[bp] = 1;
                    ++nacc;
                }
                const int left = nm - nacc;
                sel_status = left == 0 ? EB_STOP_COMPLETE : (at_cap ? EB_STOP_CAP : EB_RUNNING);
                sel_committed = nacc + (left > 0 && at_cap ? left : 0);
            }
        } else if (lane == 0) {
            sel_flag = kSelGeneral;          // more than 32 candidates: the whole CTA sorts them
            sel_ns = ns;
            sel_nm = nm;
            sel_bigmin = bigmin;
            sel_cap = at_cap ? 1 : 0;
        }
    }
    __syncthreads();
    const int flag = sel_flag;
    const bool stop = sel_stop != 0;
    if (flag & 3) {
        // non-finite logits or a wait that gave up: the canvas halts with nothing committed
        if (tid == 0) {
            a.status[b] = ((flag & 1) ? EB_STATUS_NONFINITE : 0) | ((flag & 2) ? EB_STATUS_TIMEOUT : 0);
#ifdef EB_CHECKS
            if (g_check_word) a.status[b] |= EB_STATUS_CHECK;
#endif
            if (a.steps_taken) a.steps_taken[b] = step + 1;
            if (a.committed) a.committed[b] = 0;
            if (a.mean_entropy) a.mean_entropy[b] = NAN;
        }
        for (int p = tid; p < L; p += blockDim.x) a.selected[rowbase + p] = 0;
        return;
    }
    if (flag == kSelGeneral) {
        const int ns = sel_ns, nm = sel_nm;
        const unsigned long long bigmin = sel_bigmin;
        const bool at_cap = sel_cap != 0;
        // general path: the candidates gathered by atomics, a bitonic sort in shared memory
        if (tid == 0) n_acc = 0;
        for (int p = tid; p < L; p += blockDim.x) {
            if (Ms[p] && (long long)Hq[p] <= a.bound_q) {
                const int i = atomicAdd(&n_gather, 1);
                if (EB_CHECK(i < kMaxL, kCheckRow)) keys[i] = entropy_key(Hf[p], p);
            }
        }
        int n2 = 1;
        while (n2 < ns) n2 <<= 1;
        for (int i = ns + tid; i < n2; i += blockDim.x) keys[i] = ~0ull;
        __syncthreads();
        for (int size = 2; size <= n2; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < n2; i += blockDim.x) {
                    const int ixj = i ^ stride;
                    if (ixj > i) {
                        const unsigned long long x = keys[i], y = keys[ixj];
                        const bool up = (i & size) == 0;
                        if ((x > y) == up) {
                            keys[i] = y;
                            keys[ixj] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        // inclusive scan of the sorted fixed-point entropies (Hillis-Steele)
        for (int i = tid; i < n2; i += blockDim.x) {
            const int pk = i < ns ? (int)(keys[i] & 0xFFFFFFFFu) : -1;
            scanbuf[i] = i < ns && EB_CHECK(pk >= 0 && pk < L, kCheckRow) ? Hq[pk] : 0ull;
        }
        __syncthreads();
        for (int off = 1; off < n2; off <<= 1) {
            unsigned long long add[kMaxL / kK2Threads];
            int q = 0;
            for (int i = tid; i < n2; i += blockDim.x, ++q) add[q] = i >= off ? scanbuf[i - off] : 0ull;
            __syncthreads();
            q = 0;
            for (int i = tid; i < n2; i += blockDim.x, ++q) scanbuf[i] += add[q];
            __syncthreads();
        }
        int my_acc = 0, my_rej = 0;
        for (int i = tid; i < ns; i += blockDim.x) {
            const unsigned long long excl = i == 0 ? 0ull : scanbuf[i - 1];
            if (i == 0 || (long long)excl <= a.bound_q) {
                const int pk = (int)(keys[i] & 0xFFFFFFFFu);
                if (EB_CHECK(pk >= 0 && pk < L, kCheckRow)) Acc[pk] = 1;
                ++my_acc;
            } else {
                my_rej = 1;
            }
        }
        if (my_acc) atomicAdd(&n_acc, my_acc);
        const bool all_acc = __syncthreads_or(my_rej) == 0;
        if (tid == 0) {
            int nacc = n_acc;
            if (bigmin != ~0ull && all_acc && (long long)scanbuf[ns - 1] <= a.bound_q) {
                const int bp = (int)(bigmin & 0xFFFFFFFFu);
                if (EB_CHECK(bp >= 0 && bp < L, kCheckRow)) Acc[bp] = 1;
                ++nacc;
            }
            const int left = nm - nacc;
            sel_status = left == 0 ? EB_STOP_COMPLETE : (at_cap ? EB_STOP_CAP : EB_RUNNING);
            sel_committed = nacc + (left > 0 && at_cap ? left : 0);
        }
        __syncthreads();
    }

    // 3. commit, re-mask, complete / cap
    const int new_status = sel_status;
    const float mean = sel_mean;
    for (int p = tid; p < L; p += blockDim.x) {
        const long long r = rowbase + p;
        uint8_t sel = 0;
        if (stop ? Ms[p] : Acc[p]) {
            a.tokens[r] = (stop && !a.finalize_sampled) ? As[p] : Ys[p];
            a.mask[r] = 0;
            sel = 1;
        } else if (Ms[p] && new_status == EB_STOP_CAP) {
            a.tokens[r] = a.finalize_sampled ? Ys[p] : As[p];
            a.mask[r] = 0;
            sel = 1;
        }
        a.selected[r] = sel;
        a.prev_argmax[r] = As[p];
    }
    if (tid == 0) {
        const int committed = sel_committed;
        if (new_status != EB_RUNNING) {
            a.status[b] = new_status;
            if (a.steps_taken) a.steps_taken[b] = step + 1;
        }
        if (a.committed) a.committed[b] = committed;
        if (a.mean_entropy) a.mean_entropy[b] = mean;
        if (a.committed_hist) a.committed_hist[(long long)b * a.max_steps + step] = committed;
        if (a.mean_hist) a.mean_hist[(long long)b * a.max_steps + step] = mean;
#ifdef EB_CHECKS
        __threadfence();
        if (g_check_word) a.status[b] |= EB_STATUS_CHECK;
#endif
    }
}

}  // namespace ebk

// the fused unembedding kernel reuses the partial-state helpers above
#include "eb_unembed.cuh"

// ====================================================================== host side

namespace {

thread_local std::string g_last_error;

// A named NVTX range for the lifetime of the object: every C-ABI entry point and every step of
// the loops opens one, so that a profiler's timeline shows the library's calls and steps.
// Without an attached tool the NVTX calls return at once.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
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

// Per-device launch geometry, filled once per device.
struct DeviceGeometry {
    std::atomic<int> ready{0};
    int grid[ebk::kKinds] = {};   // CTAs of k1 for each element kind
};
DeviceGeometry g_geometry[64];

template <typename K>
int resident_ctas(K kernel, int threads, size_t smem, int nsm)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const long long g = (long long)nsm * per_sm;
    return (int)(g > ebk::kMaxGrid ? ebk::kMaxGrid : g);
}

eb_status geometry(int *grid_out, int kind)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(EB_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 64) return fail(EB_ERR_UNSUPPORTED, "device index %d >= 64", dev);
    DeviceGeometry &g = g_geometry[dev];
    if (g.ready.load(std::memory_order_acquire) == 0) {
        int nsm = 0, smem_optin = 0;
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return fail(EB_ERR_CUDA, "cudaDeviceGetAttribute failed");
        if ((cudaFuncSetAttribute(ebk::k1_rowstats_direct<ebk::kF32Vec, ebk::kDirectU>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, ebk::kDirectStageBytes) != cudaSuccess ||
             cudaFuncSetAttribute(ebk::k1_rowstats_direct<ebk::kBF16Vec, ebk::kDirectU>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, ebk::kDirectStageBytes) != cudaSuccess ||
             cudaFuncSetAttribute(ebk::k1_rowstats_direct<ebk::kFP8Vec, ebk::kFP8U>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, ebk::kDirectStageBytes) != cudaSuccess ||
             cudaFuncSetAttribute(ebk::k2_select, cudaFuncAttributeMaxDynamicSharedMemorySize, ebk::kK2StageBytes) !=
                 cudaSuccess))
            return fail(EB_ERR_CUDA, "cudaFuncSetAttribute failed");
        (void)smem_optin;
        // one CTA of kDirectWarps warps per SM; every warp is one unit of the row partition
        g.grid[ebk::kF32Vec] = nsm * ebk::kDirectWarps;
        g.grid[ebk::kBF16Vec] = nsm * ebk::kDirectWarps;
        g.grid[ebk::kFP8Vec] = nsm * ebk::kDirectWarps;
        g.grid[ebk::kF32Scalar] = resident_ctas(ebk::k1_rowstats_scalar<ebk::kF32Scalar>, ebk::kConsumers, 0, nsm);
        g.grid[ebk::kBF16Scalar] = resident_ctas(ebk::k1_rowstats_scalar<ebk::kBF16Scalar>, ebk::kConsumers, 0, nsm);
        g.grid[ebk::kFP8Scalar] = resident_ctas(ebk::k1_rowstats_scalar<ebk::kFP8Scalar>, ebk::kConsumers, 0, nsm);
        g.ready.store(1, std::memory_order_release);
    }
    *grid_out = g.grid[kind];
    return EB_OK;
}

// Per-device set-up of the fused unembedding kernel: SM count and its shared-memory limit.
struct UnembedGeometry {
    std::atomic<int> ready{0};
    int nsm = 0;
};
UnembedGeometry g_unembed[64];

eb_status unembed_geometry(int *nsm_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(EB_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 64) return fail(EB_ERR_UNSUPPORTED, "device index %d >= 64", dev);
    UnembedGeometry &g = g_unembed[dev];
    if (g.ready.load(std::memory_order_acquire) == 0) {
        int nsm = 0, smem_optin = 0, major = 0;
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
            return fail(EB_ERR_CUDA, "cudaDeviceGetAttribute failed");
        if (major != 10) return fail(EB_ERR_UNSUPPORTED, "the fused unembedding kernel needs tcgen05 (sm_10x)");
        const size_t smem = ebk::k3::Smem::alloc;
        if ((size_t)smem_optin < smem)
            return fail(EB_ERR_UNSUPPORTED, "device offers %d B of shared memory per block, need %zu",
                        smem_optin, smem);
        if (cudaFuncSetAttribute(ebk::k3::k3_unembed<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(ebk::k3::k3_unembed<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(ebk::k2_select, cudaFuncAttributeMaxDynamicSharedMemorySize, ebk::kK2StageBytes) !=
                cudaSuccess)
            return fail(EB_ERR_CUDA, "cudaFuncSetAttribute failed");
        g.nsm = nsm;
        g.ready.store(1, std::memory_order_release);
    }
    *nsm_out = g.nsm;
    return EB_OK;
}

// cuTensorMapEncodeTiled from the driver (looked up once through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// 2-D bf16 tensor map of a row-major [outer, inner] matrix (inner contiguous) with a
// box_inner x box_outer box and 128-byte swizzle; out-of-range elements read as zero.
eb_status encode_bf16_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                         uint32_t box_outer)
{
    EncodeTiledFn f = encode_fn();
    if (!f) return fail(EB_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(EB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return EB_OK;
}

// Records a profiling event on `stream`; inside a stream capture it becomes a real event
// record node of the graph (so the event can time each replay).
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    return cudaEventRecord(ev, stream);
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

// Workspace layout: [partials (rows + kMaxGrid) x 32 B][weight prefix (rows + 1) x 4 B]
// [first / last partition unit of each row, rows x 8 B], each part 256-byte aligned.
constexpr size_t align256c(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t partial_bytes(long long rows) { return align256c((size_t)(rows + ebk::kMaxGrid) * sizeof(ebk::Partial)); }
constexpr size_t prefix_bytes(long long rows) { return align256c((size_t)(rows + 1) * sizeof(uint32_t)); }
constexpr size_t rowunit_bytes(long long rows) { return align256c((size_t)rows * sizeof(int2)); }
constexpr size_t pass_workspace_bytes(long long rows)
{
    return partial_bytes(rows) + prefix_bytes(rows) + rowunit_bytes(rows);
}
// Two copies: the step's row statistics, and the raw-logit pass of EB_FLAG_STOP_RAW_ENTROPY.
constexpr size_t step_workspace_bytes(long long rows) { return 2 * pass_workspace_bytes(rows); }

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
    // continuous batching: per-canvas step, Philox canvas id, c and 1/T (all or none)
    const int32_t *canvas_step = nullptr;
    const int32_t *canvas_id = nullptr;
    const float *canvas_c = nullptr;
    const float *canvas_invT = nullptr;
};

eb_status check_common(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                       const void *d_logits, const StepBuffers &sb, void *d_ws, size_t ws_bytes,
                       size_t ws_needed)
{
    if (!params) return fail(EB_ERR_INVALID, "params is NULL");
    if ((params->flags & ~(uint32_t)(EB_FLAG_DIAG_STALL | EB_FLAG_STOP_MASKED_ONLY | EB_FLAG_FINALIZE_SAMPLED |
                                     EB_FLAG_STOP_RAW_ENTROPY)) != 0)
        return fail(EB_ERR_INVALID, "params->flags has unknown bits 0x%x", params->flags);
    if (params->max_steps < 1) return fail(EB_ERR_INVALID, "max_steps must be >= 1");
    if (!(params->t_start > 0.0f) || !(params->t_end > 0.0f) || !std::isfinite(params->t_start) ||
        !std::isfinite(params->t_end))
        return fail(EB_ERR_INVALID, "temperatures must be finite and > 0");
    if (!std::isfinite(params->entropy_bound) || !std::isfinite(params->stop_entropy) ||
        std::fabs(params->entropy_bound) > 1.0e6f || std::fabs(params->stop_entropy) > 1.0e6f)
        return fail(EB_ERR_INVALID, "entropy_bound / stop_entropy must be finite and below 1e6");
    if (B < 0) return fail(EB_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (L < 1 || L > ebk::kMaxL) return fail(EB_ERR_INVALID, "L must be in [1, %d] (got %d)", ebk::kMaxL, L);
    if (V < 1) return fail(EB_ERR_INVALID, "V must be >= 1 (got %d)", V);
    if (dtype != EB_F32 && dtype != EB_BF16 && dtype != EB_FP8_E4M3)
        return fail(EB_ERR_INVALID, "unknown dtype %d", (int)dtype);
    if (B == 0) return EB_OK;
    if (!d_logits) return fail(EB_ERR_INVALID, "d_logits is NULL");
    if (!sb.mask || !sb.tokens || !sb.prev_argmax || !sb.status || !sb.entropy || !sb.argmax ||
        !sb.sampled || !sb.selected)
        return fail(EB_ERR_INVALID, "a required state / output pointer is NULL");
    const long long rows = (long long)B * L;
    if (rows > (1ll << 31) - 1 - ebk::kMaxGrid) return fail(EB_ERR_UNSUPPORTED, "B*L too large");
    if (!d_ws) return fail(EB_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)d_ws & 255) != 0) return fail(EB_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < ws_needed)
        return fail(EB_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, ws_needed);
    return EB_OK;
}

struct RawPass {                 // partial states of the raw-logit pass, or all null
    const ebk::Partial *partials = nullptr;
    const uint32_t *prefix = nullptr;
    const int2 *rowunits = nullptr;
    int G = 0, weighted = 0;
};

// Enqueues the selection kernel over the partial states of this step (and of the raw-logit
// pass, when given) as a programmatic dependent of the row-statistics grid.
eb_status launch_select(const eb_params *params, int B, int L, int step, float c, const StepBuffers &sb,
                        const ebk::Partial *partials, const uint32_t *prefix, const int2 *rowunits,
                        long long nvec_row,
                        int rows, int G, int weighted, int k3_g, cudaStream_t stream,
                        const RawPass &raw = RawPass())
{
    ebk::K2Args a2;
#ifdef EB_CHECKS
    // partial-state slots: the streaming layout, or the fused kernel's (row block, group rank,
    // column group, row) layout
    a2.nslots = k3_g > 0 ? (long long)((rows + ebk::k3::BM - 1) / ebk::k3::BM) * k3_g * ebk::k3::kEpiGroups * ebk::k3::BM
                         : (long long)rows + ebk::kMaxGrid;
#endif
    a2.partials = partials;
    a2.prefix = prefix;
    a2.rowunits = rowunits;
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
    a2.rows = rows;
    a2.L = L;
    a2.G = G;
    a2.step = step;
    a2.max_steps = params->max_steps;
    a2.weighted = weighted;
    a2.c = c;
    // fixed point, 2^-40 nats: accept while prefix <= floor(bound), stop while sum < ceil(stop L)
    a2.bound_q = (long long)std::floor((double)params->entropy_bound * 1099511627776.0);
    a2.stop_q = (long long)std::ceil((double)params->stop_entropy * (double)L * 1099511627776.0);
    a2.stop_entropy = (double)params->stop_entropy;
    a2.canvas_step = sb.canvas_step;
    a2.canvas_c = sb.canvas_c;
    a2.raw_partials = raw.partials;
    a2.raw_prefix = raw.prefix;
    a2.raw_rowunits = raw.rowunits;
    a2.raw_G = raw.G;
    a2.raw_weighted = raw.weighted;
    a2.stop_masked_only = (params->flags & EB_FLAG_STOP_MASKED_ONLY) ? 1 : 0;
    a2.finalize_sampled = (params->flags & EB_FLAG_FINALIZE_SAMPLED) ? 1 : 0;
    a2.k3_g = k3_g;
    a2.k3_groups = ebk::k3::kEpiGroups;
    // programmatic dependent launch: the selection grid is set up while the row-statistics
    // grid drains; its griddepcontrol.wait orders the reads of the partial states
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(ebk::kK2Threads);
    cfg.dynamicSmemBytes = ebk::kK2StageBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ebk::k2_select, a2);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "selection launch: %s", cudaGetErrorString(e));
    return EB_OK;
}

// Enqueues k1 + k2 for one step.  Arguments were validated by the caller.
// One row-statistics launch of element kind `kind` over G partition units.
eb_status launch_k1(int kind, int G, const ebk::K1Args &a1, cudaStream_t stream)
{
    switch (kind) {
    // G counts warps (partition units); whole CTAs of kDirectWarps warps, the tail ones idle
    case ebk::kF32Vec:
        ebk::k1_rowstats_direct<ebk::kF32Vec, ebk::kDirectU>
            <<<(G + ebk::kDirectWarps - 1) / ebk::kDirectWarps, ebk::kDirectThreads, ebk::kDirectStageBytes, stream>>>(a1);
        break;
    case ebk::kBF16Vec:
        ebk::k1_rowstats_direct<ebk::kBF16Vec, ebk::kDirectU>
            <<<(G + ebk::kDirectWarps - 1) / ebk::kDirectWarps, ebk::kDirectThreads, ebk::kDirectStageBytes, stream>>>(a1);
        break;
    case ebk::kFP8Vec:
        ebk::k1_rowstats_direct<ebk::kFP8Vec, ebk::kFP8U>
            <<<(G + ebk::kDirectWarps - 1) / ebk::kDirectWarps, ebk::kDirectThreads, ebk::kDirectStageBytes, stream>>>(a1);
        break;
    case ebk::kF32Scalar: ebk::k1_rowstats_scalar<ebk::kF32Scalar><<<G, ebk::kConsumers, 0, stream>>>(a1); break;
    case ebk::kBF16Scalar: ebk::k1_rowstats_scalar<ebk::kBF16Scalar><<<G, ebk::kConsumers, 0, stream>>>(a1); break;
    default: ebk::k1_rowstats_scalar<ebk::kFP8Scalar><<<G, ebk::kConsumers, 0, stream>>>(a1); break;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "row-statistics launch: %s", cudaGetErrorString(e));
    return EB_OK;
}

eb_status launch_step(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                      const void *d_logits, int step, float T, const StepBuffers &sb,
                      void *d_ws, cudaStream_t stream)
{
    const size_t esize = dtype == EB_F32 ? 4 : (dtype == EB_BF16 ? 2 : 1);
    const bool aligned = (((uintptr_t)d_logits & 15) == 0) && (((size_t)V * esize) % 16 == 0);
    int kind;
    if (dtype == EB_F32) kind = aligned ? ebk::kF32Vec : ebk::kF32Scalar;
    else if (dtype == EB_BF16) kind = aligned ? ebk::kBF16Vec : ebk::kBF16Scalar;
    else kind = aligned ? ebk::kFP8Vec : ebk::kFP8Scalar;
    const int vec = aligned ? (int)(16 / esize) : 1;
    int gmax = 0;
    eb_status st = geometry(&gmax, kind);
    if (st != EB_OK) return st;
    const long long rows = (long long)B * L;
    const long long nvec_row = V / vec;
    const long long N = rows * nvec_row;
    if (N > (1ll << 48)) return fail(EB_ERR_UNSUPPORTED, "B*L*V too large");
    const bool weighted = rows <= ebk::kMaxWeightedRows &&
                          (unsigned long long)N * ebk::kWeightMasked < (1ull << 32);
    const int G = (int)(N < gmax ? N : gmax);
    char *ws = static_cast<char *>(d_ws);
    ebk::Partial *partials = reinterpret_cast<ebk::Partial *>(ws);
    uint32_t *prefix = reinterpret_cast<uint32_t *>(ws + partial_bytes(rows));
    int2 *rowunits = reinterpret_cast<int2 *>(ws + partial_bytes(rows) + prefix_bytes(rows));

    ebk::K1Args a1;
    a1.logits = d_logits;
    a1.mask = sb.mask;
    a1.status = sb.status;
    a1.partials = partials;
    a1.prefix_out = prefix;
    a1.rowunits = rowunits;
    a1.nvec_row = nvec_row;
    a1.row_bytes = (long long)V * (long long)esize;
    a1.rows = (int)rows;
    a1.L = L;
    a1.G = G;
    a1.step = step;
    a1.weighted = weighted ? 1 : 0;
    a1.c = ebk::kLog2e / T;
    a1.invT = 1.0f / T;
    a1.keys = round_keys(params->seed);
    a1.canvas_step = sb.canvas_step;
    a1.canvas_id = sb.canvas_id;
    a1.canvas_c = sb.canvas_c;
    a1.canvas_invT = sb.canvas_invT;
    a1.raw = 0;
#ifdef EB_CHECKS
    a1.nslots = rows + ebk::kMaxGrid;
#endif
    // EB_FLAG_STOP_RAW_ENTROPY: first a pass at T = 1 with every row unmasked (no sampling)
    // into the second workspace copy; the selection kernel sums its entropies for the stop rule
    RawPass raw;
    if (params->flags & EB_FLAG_STOP_RAW_ENTROPY) {
        ebk::K1Args ar = a1;
        char *wr = ws + pass_workspace_bytes(rows);
        ar.partials = reinterpret_cast<ebk::Partial *>(wr);
        ar.prefix_out = reinterpret_cast<uint32_t *>(wr + partial_bytes(rows));
        ar.rowunits = reinterpret_cast<int2 *>(wr + partial_bytes(rows) + prefix_bytes(rows));
        ar.c = ebk::kLog2e;
        ar.invT = 1.0f;
        ar.canvas_step = nullptr;
        ar.canvas_id = nullptr;
        ar.canvas_c = nullptr;
        ar.canvas_invT = nullptr;
        ar.raw = 1;
        st = launch_k1(kind, G, ar, stream);
        if (st != EB_OK) return st;
        raw.partials = ar.partials;
        raw.prefix = ar.prefix_out;
        raw.rowunits = ar.rowunits;
        raw.G = G;
        raw.weighted = ar.weighted;
    }
    cudaEvent_t prof_begin = g_profile_begin, prof_end = g_profile_end;
    g_profile_begin = g_profile_end = nullptr;
    if (prof_begin && record_profile_event(prof_begin, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");
    st = launch_k1(kind, G, a1, stream);
    if (st != EB_OK) return st;
    if (prof_end && record_profile_event(prof_end, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");

    return launch_select(params, B, L, step, a1.c, sb, partials, prefix, rowunits, nvec_row, (int)rows, G,
                         a1.weighted, 0, stream, raw);
}

// Enqueues the fused unembedding kernel (+ the selection kernel unless logits_out is given).
// Arguments were validated by the caller.
eb_status launch_unembed(const eb_params *params, int B, int L, int K, int V, const void *d_h,
                         const void *d_W, int step, float T, const StepBuffers *sb, void *d_ws,
                         float *logits_out, cudaStream_t stream)
{
    namespace k3 = ebk::k3;
    if (params && (params->flags & EB_FLAG_STOP_RAW_ENTROPY))
        return fail(EB_ERR_UNSUPPORTED, "EB_FLAG_STOP_RAW_ENTROPY needs the logits twice; the fused path never stores them");
    int nsm = 0;
    eb_status st = unembed_geometry(&nsm);
    if (st != EB_OK) return st;
    const long long M = (long long)B * L;
    const int MB = (int)((M + k3::BM - 1) / k3::BM);
    const int NB = (int)(((long long)V + k3::BN - 1) / k3::BN);
    const int KB = (K + k3::BK - 1) / k3::BK;
    const int Gmax = nsm < k3::kMaxCtas ? nsm : k3::kMaxCtas;
    int g, G;
    if (MB <= Gmax) {
        g = Gmax / MB;
        if (g > NB) g = NB;
        G = MB * g;
    } else {
        g = 1;
        G = Gmax;
    }
    CUtensorMap th, tw;
    st = encode_bf16_2d(&th, d_h, (uint64_t)K, (uint64_t)M, k3::BK, k3::BM);
    if (st != EB_OK) return st;
    st = encode_bf16_2d(&tw, d_W, (uint64_t)V, (uint64_t)K, 64, k3::BK);
    if (st != EB_OK) return st;

    k3::Args a;
    a.mask = sb ? sb->mask : nullptr;
    a.status = sb ? sb->status : nullptr;
    a.partials = static_cast<ebk::Partial *>(d_ws);
    a.logits = logits_out;
    a.M = (int)M;
    a.K = K;
    a.V = V;
    a.L = L;
    a.MB = MB;
    a.NB = NB;
    a.KB = KB;
    a.g = g;
    a.G = G;
    a.step = step;
    a.c = ebk::kLog2e / T;
    a.invT = 1.0f / T;
    a.keys = round_keys(params ? params->seed : 0);
    a.stall_first = (params && (params->flags & EB_FLAG_DIAG_STALL)) ? 1 : 0;
    a.wait_limit = a.stall_first ? ebk::kDiagWaitLimit : ebk::kWaitLimit;
    cudaEvent_t prof_begin = g_profile_begin, prof_end = g_profile_end;
    g_profile_begin = g_profile_end = nullptr;
    if (prof_begin && record_profile_event(prof_begin, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");
    if (logits_out)
        k3::k3_unembed<true><<<G, k3::kThreads, k3::Smem::alloc, stream>>>(th, tw, a);
    else
        k3::k3_unembed<false><<<G, k3::kThreads, k3::Smem::alloc, stream>>>(th, tw, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "unembedding launch: %s", cudaGetErrorString(e));
    if (prof_end && record_profile_event(prof_end, stream) != cudaSuccess)
        return fail(EB_ERR_CUDA, "cudaEventRecord failed");
    if (logits_out) return EB_OK;
    return launch_select(params, B, L, step, a.c, *sb, a.partials, nullptr, nullptr, 0, (int)M, G, 0, g, stream);
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
    return step_workspace_bytes((long long)B * L);
}

eb_status eb_sampler_step(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                          const void *d_logits, int step, float temperature,
                          uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                          int32_t *d_status, int32_t *d_steps_taken,
                          float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                          uint8_t *d_selected, int32_t *d_committed, float *d_mean_entropy,
                          void *d_workspace, size_t workspace_bytes, void *stream)
{
    NvtxRange range("eb_sampler_step");
    StepBuffers sb{d_mask, d_tokens, d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax,
                   d_sampled, d_selected, d_committed, d_mean_entropy, nullptr, nullptr};
    eb_status st = check_common(params, B, L, V, dtype, d_logits, sb, d_workspace, workspace_bytes,
                                eb_workspace_bytes(B, L, V, dtype));
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

}  // extern "C"

// ---------------------------------------------------------------- fixed-scratch variant
//
// Scratch of eb_sampler_step_noalloc: a file-scope device array sized for at most
// EB_NOALLOC_MAX_ROWS canvas positions (B * L).  Every device that loads this library holds
// it until the process exits.  Host code cannot use the array's name as a device address,
// so its address is looked up once per device with cudaGetSymbolAddress and cached.
namespace {

constexpr long long kNoallocRows = EB_NOALLOC_MAX_ROWS;
constexpr size_t kNoallocBytes = step_workspace_bytes(kNoallocRows);

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

namespace {

// The array's device address per device ordinal, null until the first call on that device.
// Two threads that make the first call at once both look it up and store the same value.
std::atomic<void *> g_noalloc[64];

// Device address of the array on the current device (set up on the first call per device).
eb_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(EB_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= 64) return fail(EB_ERR_UNSUPPORTED, "device index %d >= 64", dev);
    void *p = g_noalloc[dev].load(std::memory_order_acquire);
    if (!p) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(EB_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch: %s", cudaGetErrorString(e));
        g_noalloc[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return EB_OK;
}

}  // namespace

extern "C" {

eb_status eb_sampler_step_noalloc(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                                  const void *d_logits, int step, float temperature,
                                  uint8_t *d_mask, int32_t *d_tokens, int32_t *d_prev_argmax,
                                  int32_t *d_status, int32_t *d_steps_taken,
                                  float *d_entropy, int32_t *d_argmax, int32_t *d_sampled,
                                  uint8_t *d_selected, int32_t *d_committed, float *d_mean_entropy,
                                  void *stream)
{
    NvtxRange range("eb_sampler_step_noalloc");
    if (B > 0 && L > 0 && (long long)B * L > kNoallocRows)
        return fail(EB_ERR_UNSUPPORTED, "B*L = %lld exceeds the fixed scratch of %lld positions; use "
                    "eb_sampler_step with a caller-allocated workspace", (long long)B * L, kNoallocRows);
    void *scratch = nullptr;
    if (B > 0) {
        const eb_status st = noalloc_scratch(&scratch);
        if (st != EB_OK) return st;
        if (eb_workspace_bytes(B, L, V, dtype) > kNoallocBytes)
            return fail(EB_ERR_UNSUPPORTED, "the fixed scratch is too small for this call");
    }
    return eb_sampler_step(params, B, L, V, dtype, d_logits, step, temperature, d_mask, d_tokens,
                           d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax, d_sampled,
                           d_selected, d_committed, d_mean_entropy, scratch, kNoallocBytes, stream);
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
    NvtxRange range("eb_sample_canvas");
    if (steps_run) *steps_run = 0;
    StepBuffers sb{d_mask, d_tokens, d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax,
                   d_sampled, d_selected, nullptr, nullptr, d_committed_per_step,
                   d_mean_entropy_per_step};
    eb_status st = check_common(params, B, L, V, dtype, d_logits, sb, d_workspace, workspace_bytes,
                                eb_workspace_bytes(B, L, V, dtype));
    if (st != EB_OK) return st;
    if (!logits_fn) return fail(EB_ERR_INVALID, "logits_fn is NULL");
    if (start_step < 0) return fail(EB_ERR_INVALID, "start_step must be >= 0");
    if (poll_every < 0) return fail(EB_ERR_INVALID, "poll_every must be >= 0");
    if (B == 0) return ok();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int ran = 0;
    for (int step = start_step; step < params->max_steps; ++step) {
        NvtxRange step_range("eb_sample_canvas step");
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

}  // extern "C"

// ---------------------------------------------------------------- block driver
//
// Continuous batching over B canvas slots: block k of n is a fresh all-masked canvas whose
// Philox canvas id is k.  Every iteration the denoiser fills the logits of the occupied slots,
// one sampler step runs with each slot's own step and temperature, and the refill kernel
// retires the slots that stopped (their tokens, step count and stop reason go to block k's
// outputs) and hands them the next block, or leaves them idle when none is left.
namespace {

struct BlockSlots {
    uint8_t *mask;
    int32_t *tokens, *prev_argmax, *status, *steps_taken;
    float *entropy;
    int32_t *argmax, *sampled;
    uint8_t *selected;
    int32_t *slot_block, *slot_step;
    float *slot_c, *slot_invT;
    int32_t *counters;          // [0] next block to hand out, [1] blocks finished
};

// The schedule temperature of `step` and its c = log2(e) / T and 1 / T, with the same binary32
// operations, in the same order, as the host's eb_temperature (no contraction).
__device__ __forceinline__ void slot_temperature(float t_start, float t_end, int max_steps, int step,
                                                 float *c, float *invT)
{
    float T = t_start;
    if (max_steps > 1)
        T = __fadd_rn(t_start, __fdiv_rn(__fmul_rn(__fsub_rn(t_end, t_start), (float)step), (float)(max_steps - 1)));
    *c = __fdiv_rn(ebk::kLog2e, T);
    *invT = __fdiv_rn(1.0f, T);
}

__device__ void slot_reset(const BlockSlots &s, int b, int L, int block, float t_start, float t_end,
                           int max_steps)
{
    const long long base = (long long)b * L;
    for (int p = threadIdx.x; p < L; p += blockDim.x) {
        s.mask[base + p] = block >= 0 ? 1 : 0;
        s.tokens[base + p] = -1;
        s.prev_argmax[base + p] = -1;
    }
    if (threadIdx.x == 0) {
        s.status[b] = block >= 0 ? EB_RUNNING : EB_SLOT_IDLE;
        s.steps_taken[b] = 0;
        s.slot_block[b] = block;
        s.slot_step[b] = 0;
        slot_temperature(t_start, t_end, max_steps, 0, &s.slot_c[b], &s.slot_invT[b]);
    }
}

__global__ void blocks_init(const BlockSlots s, int L, int n_blocks, float t_start, float t_end, int max_steps)
{
    const int b = blockIdx.x;
    slot_reset(s, b, L, b < n_blocks ? b : -1, t_start, t_end, max_steps);
    if (b == 0 && threadIdx.x == 0) {
        s.counters[0] = (int)gridDim.x < n_blocks ? (int)gridDim.x : n_blocks;
        s.counters[1] = 0;
    }
}

// One CTA per slot, after the sampler step of an iteration.
__global__ void blocks_refill(const BlockSlots s, int L, int n_blocks, int32_t *block_tokens,
                              int32_t *block_steps, int32_t *block_status, float t_start, float t_end,
                              int max_steps)
{
    __shared__ int next;
    const int b = blockIdx.x;
    const int k = s.slot_block[b];
    if (k < 0) return;                               // idle slot (CTA-uniform)
    const int st = s.status[b];
    if (st == EB_RUNNING) {
        if (threadIdx.x == 0) {
            const int step = s.slot_step[b] + 1;
            s.slot_step[b] = step;
            slot_temperature(t_start, t_end, max_steps, step, &s.slot_c[b], &s.slot_invT[b]);
        }
        return;
    }
    const long long base = (long long)b * L, out = (long long)k * L;
    for (int p = threadIdx.x; p < L; p += blockDim.x) block_tokens[out + p] = s.tokens[base + p];
    if (threadIdx.x == 0) {
        if (block_steps) block_steps[k] = s.steps_taken[b];
        if (block_status) block_status[k] = st;
        atomicAdd(&s.counters[1], 1);
        next = atomicAdd(&s.counters[0], 1);
    }
    __syncthreads();
    slot_reset(s, b, L, next < n_blocks ? next : -1, t_start, t_end, max_steps);
}

struct BlocksLayout {
    size_t step, mask, tokens, prev, status, steps, entropy, argmax, sampled, selected, block, sstep, c,
        invT, counters, total;
};

BlocksLayout blocks_layout(int B, int L)
{
    const long long rows = (long long)B * L;
    BlocksLayout o;
    size_t at = 0;
    auto take = [&](size_t bytes) { const size_t r = at; at += align256(bytes); return r; };
    o.step = take(step_workspace_bytes(rows));
    o.mask = take((size_t)rows);
    o.tokens = take((size_t)rows * 4);
    o.prev = take((size_t)rows * 4);
    o.status = take((size_t)B * 4);
    o.steps = take((size_t)B * 4);
    o.entropy = take((size_t)rows * 4);
    o.argmax = take((size_t)rows * 4);
    o.sampled = take((size_t)rows * 4);
    o.selected = take((size_t)rows);
    o.block = take((size_t)B * 4);
    o.sstep = take((size_t)B * 4);
    o.c = take((size_t)B * 4);
    o.invT = take((size_t)B * 4);
    o.counters = take(16);
    o.total = at;
    return o;
}

}  // namespace

extern "C" {

size_t eb_blocks_workspace_bytes(int B, int L, int V, eb_dtype dtype)
{
    (void)V;
    (void)dtype;
    if (B < 1 || L < 1) return 0;
    return blocks_layout(B, L).total;
}

eb_status eb_sample_blocks(const eb_params *params, int B, int L, int V, eb_dtype dtype,
                           eb_block_logits_fn logits_fn, void *user, void *d_logits, int n_blocks,
                           int32_t *d_block_tokens, int32_t *d_block_steps, int32_t *d_block_status,
                           void *d_workspace, size_t workspace_bytes, int poll_every, int *iterations_run,
                           void *stream)
{
    NvtxRange range("eb_sample_blocks");
    if (iterations_run) *iterations_run = 0;
    if (!params) return fail(EB_ERR_INVALID, "params is NULL");
    if (B < 1) return fail(EB_ERR_INVALID, "B must be >= 1 slot");
    if (n_blocks < 0 || n_blocks > (1 << 24)) return fail(EB_ERR_INVALID, "n_blocks must be in [0, 2^24]");
    if (!logits_fn) return fail(EB_ERR_INVALID, "logits_fn is NULL");
    if (!d_block_tokens && n_blocks > 0) return fail(EB_ERR_INVALID, "d_block_tokens is NULL");
    if (poll_every < 0) return fail(EB_ERR_INVALID, "poll_every must be >= 0");
    const size_t need = eb_blocks_workspace_bytes(B, L, V, dtype);
    char *ws = static_cast<char *>(d_workspace);
    if (!ws || ((uintptr_t)ws & 255) != 0 || workspace_bytes < need)
        return fail(EB_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
    const BlocksLayout o = blocks_layout(B, L);
    BlockSlots sl;
    sl.mask = reinterpret_cast<uint8_t *>(ws + o.mask);
    sl.tokens = reinterpret_cast<int32_t *>(ws + o.tokens);
    sl.prev_argmax = reinterpret_cast<int32_t *>(ws + o.prev);
    sl.status = reinterpret_cast<int32_t *>(ws + o.status);
    sl.steps_taken = reinterpret_cast<int32_t *>(ws + o.steps);
    sl.entropy = reinterpret_cast<float *>(ws + o.entropy);
    sl.argmax = reinterpret_cast<int32_t *>(ws + o.argmax);
    sl.sampled = reinterpret_cast<int32_t *>(ws + o.sampled);
    sl.selected = reinterpret_cast<uint8_t *>(ws + o.selected);
    sl.slot_block = reinterpret_cast<int32_t *>(ws + o.block);
    sl.slot_step = reinterpret_cast<int32_t *>(ws + o.sstep);
    sl.slot_c = reinterpret_cast<float *>(ws + o.c);
    sl.slot_invT = reinterpret_cast<float *>(ws + o.invT);
    sl.counters = reinterpret_cast<int32_t *>(ws + o.counters);
    StepBuffers sb{sl.mask, sl.tokens, sl.prev_argmax, sl.status, sl.steps_taken, sl.entropy, sl.argmax,
                   sl.sampled, sl.selected, nullptr, nullptr, nullptr, nullptr};
    sb.canvas_step = sl.slot_step;
    sb.canvas_id = sl.slot_block;
    sb.canvas_c = sl.slot_c;
    sb.canvas_invT = sl.slot_invT;
    eb_status st = check_common(params, B, L, V, dtype, d_logits, sb, ws + o.step, o.mask - o.step,
                                eb_workspace_bytes(B, L, V, dtype));
    if (st != EB_OK) return st;
    if (n_blocks == 0) return ok();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    blocks_init<<<B, 256, 0, s>>>(sl, L, n_blocks, params->t_start, params->t_end, params->max_steps);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(EB_ERR_CUDA, "block set-up launch: %s", cudaGetErrorString(e));
    // every iteration advances every occupied slot by one step, so n_blocks * max_steps
    // iterations finish any schedule; the host stops earlier once the finished count is n_blocks
    const long long max_iter = (long long)n_blocks * params->max_steps;
    int ran = 0;
    for (long long it = 0; it < max_iter; ++it) {
        NvtxRange iter_range("eb_sample_blocks iteration");
        if (poll_every > 0 && it > 0 && it % poll_every == 0) {
            int32_t done = 0;
            e = cudaMemcpyAsync(&done, sl.counters + 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) {
                if (iterations_run) *iterations_run = ran;
                return fail(EB_ERR_CUDA, "progress read-back: %s", cudaGetErrorString(e));
            }
            if (done >= n_blocks) break;
        }
        if (logits_fn(user, B, sl.slot_block, sl.slot_step, sl.tokens, d_logits, stream) != 0) {
            if (iterations_run) *iterations_run = ran;
            return fail(EB_ERR_CALLBACK, "logits callback failed at iteration %lld", it);
        }
        st = launch_step(params, B, L, V, dtype, d_logits, 0, params->t_start, sb, ws + o.step, s);
        if (st != EB_OK) {
            if (iterations_run) *iterations_run = ran;
            return st;
        }
        blocks_refill<<<B, 256, 0, s>>>(sl, L, n_blocks, d_block_tokens, d_block_steps, d_block_status,
                                        params->t_start, params->t_end, params->max_steps);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            if (iterations_run) *iterations_run = ran;
            return fail(EB_ERR_CUDA, "refill launch: %s", cudaGetErrorString(e));
        }
        ++ran;
    }
    if (iterations_run) *iterations_run = ran;
    return ok();
}

size_t eb_unembed_workspace_bytes(int B, int L, int K, int V)
{
    (void)K;
    (void)V;
    if (B < 0 || L < 1) return 0;
    const long long M = (long long)B * L;
    const long long MB = (M + ebk::k3::BM - 1) / ebk::k3::BM;
    const long long slots = MB > ebk::k3::kMaxCtas ? MB : ebk::k3::kMaxCtas;
    return align256((size_t)slots * ebk::k3::kEpiGroups * ebk::k3::BM * sizeof(ebk::Partial));
}

namespace {

eb_status check_unembed(int M, int K, int V, const void *d_h, const void *d_W)
{
    if (M < 0) return fail(EB_ERR_INVALID, "B*L must be >= 0");
    if (K < 8 || K % 8 != 0) return fail(EB_ERR_INVALID, "K must be a positive multiple of 8 (got %d)", K);
    if (V < 8 || V % 8 != 0) return fail(EB_ERR_INVALID, "V must be a positive multiple of 8 (got %d)", V);
    if (M == 0) return EB_OK;
    if (!d_h || !d_W) return fail(EB_ERR_INVALID, "d_h / d_W is NULL");
    if (((uintptr_t)d_h & 15) || ((uintptr_t)d_W & 15))
        return fail(EB_ERR_INVALID, "d_h and d_W must be 16-byte aligned");
    return EB_OK;
}

}  // namespace

eb_status eb_unembed_sample(const eb_params *params, int B, int L, int K, int V, const void *d_h,
                            const void *d_W, int step, float temperature, uint8_t *d_mask,
                            int32_t *d_tokens, int32_t *d_prev_argmax, int32_t *d_status,
                            int32_t *d_steps_taken, float *d_entropy, int32_t *d_argmax,
                            int32_t *d_sampled, uint8_t *d_selected, int32_t *d_committed,
                            float *d_mean_entropy, void *d_workspace, size_t workspace_bytes,
                            void *stream)
{
    NvtxRange range("eb_unembed_sample");
    StepBuffers sb{d_mask, d_tokens, d_prev_argmax, d_status, d_steps_taken, d_entropy, d_argmax,
                   d_sampled, d_selected, d_committed, d_mean_entropy, nullptr, nullptr};
    eb_status st = check_common(params, B, L, V, EB_BF16, d_h, sb, d_workspace, workspace_bytes,
                                eb_unembed_workspace_bytes(B, L, K, V));
    if (st != EB_OK) return st;
    if (B == 0) return ok();
    st = check_unembed(B * L, K, V, d_h, d_W);
    if (st != EB_OK) return st;
    if (step < 0 || step >= params->max_steps)
        return fail(EB_ERR_INVALID, "step %d outside [0, max_steps=%d)", step, params->max_steps);
    if (std::isnan(temperature) || std::isinf(temperature))
        return fail(EB_ERR_INVALID, "temperature must be finite");
    const float T = temperature > 0.0f ? temperature : schedule_temperature(params, step);
    st = launch_unembed(params, B, L, K, V, d_h, d_W, step, T, &sb, d_workspace, nullptr,
                        static_cast<cudaStream_t>(stream));
    return st == EB_OK ? ok() : st;
}

eb_status eb_unembed_logits(int M, int K, int V, const void *d_h, const void *d_W, float *d_logits,
                            void *stream)
{
    NvtxRange range("eb_unembed_logits");
    eb_status st = check_unembed(M, K, V, d_h, d_W);
    if (st != EB_OK) return st;
    if (M == 0) return ok();
    if (!d_logits) return fail(EB_ERR_INVALID, "d_logits is NULL");
    if (M > (1 << 30)) return fail(EB_ERR_UNSUPPORTED, "M too large");
    // one canvas of M positions as far as the launch geometry is concerned
    st = launch_unembed(nullptr, 1, M, K, V, d_h, d_W, 0, 1.0f, nullptr, nullptr, d_logits,
                        static_cast<cudaStream_t>(stream));
    return st == EB_OK ? ok() : st;
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

int eb_checks_enabled(void)
{
#ifdef EB_CHECKS
    return 1;
#else
    return 0;
#endif
}

uint32_t eb_check_word(int clear)
{
#ifdef EB_CHECKS
    unsigned int w = 0;
    if (cudaMemcpyFromSymbol(&w, ebk::g_check_word, sizeof w) != cudaSuccess) return 0;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(ebk::g_check_word, &z, sizeof z) != cudaSuccess) return 0;
    }
    return w;
#else
    (void)clear;
    return 0;
#endif
}

}  // extern "C"
