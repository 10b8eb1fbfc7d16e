// eb_unembed.cuh -- fused unembedding GEMM + sampler row statistics for B300 (sm_103a).
//
// logits[m, v] = sum_k h[m, k] W[k, v] (bf16 inputs, fp32 accumulation) is computed tile by
// tile on the 5th-generation tensor cores, and every 128 x 256 accumulator tile is consumed in
// place by the sampler's per-row online state (max, sum 2^t, sum t 2^t, first argmax, Gumbel-max
// sample; the same state and merge as the streaming row-statistics kernel), so the logits never
// reach HBM.  The selection kernel then merges the per-CTA partial states exactly as it does for
// streamed logits.  (DiffusionGemma model card, "Best practices" section 1: the sampler consumes
// the decoder's full-vocabulary logits of every canvas position at every denoising step.)
//
// One CTA per SM, 576 threads, warp-specialised:
//   warp 0      TMA producer: per 64-wide K slice one 128 x 64 box of h (K-major, 128-byte
//               swizzle) and four 64 x 64 boxes of W (V contiguous, i.e. an N-major B operand)
//               into a 4-stage shared-memory ring, completion counted on mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and issues
//               tcgen05.mma (M=128, N=256, K=16, kind::f16, bf16 x bf16 -> fp32) from one lane;
//               tcgen05.commit releases ring stages and hands finished accumulators over;
//   warps 2..17 epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (one canvas row per thread)
//               and accumulator columns 64 ((w - 2) / 4) .. +63 with tcgen05.ld, 32 columns at
//               a time (the next load in flight while a chunk is consumed), and updates its row's
//               state in groups of 8 columns with the streaming kernel's per-group body; it frees
//               the accumulator for the next tile.
// The two accumulators let the MMA of tile i+1 run while the epilogue consumes tile i.
//
// Schedule: the M x V output is cut into MB = ceil(M/128) row blocks and NB = ceil(V/256)
// column tiles.  With MB <= G (CTAs), CTA c owns row block c % MB and column tiles j, j+g, ...
// (j = c / MB, g = G / MB), so the MB CTAs that share j read the same W tile at about the same
// time (one HBM read, the rest from L2) and each CTA keeps its rows' state in registers for its
// whole column range.  Partial state of (row block mb, group rank j, column group hh, row
// lane) lands in slot ((mb g + j) kEpiGroups + hh) 128 + lane; the selection kernel merges them
// in that order.
//
// Every mbarrier wait is bounded.  A role whose wait gives up raises a shared abort flag, the
// others leave their loops at their next wait, the producer waits (bounded) for its copies in
// flight, the MMA warp waits (bounded) for its last commit, partials are flagged, TMEM is freed
// and the CTA returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "eb_kernels.cuh"

namespace ebk {
namespace k3 {

constexpr int BM = 128;                       // rows per tile (TMEM lanes)
constexpr int BN = 256;                       // columns per tile (one accumulator)
constexpr int BK = 64;                        // K per ring stage (one 128-byte swizzle row)
constexpr int UK = 16;                        // K per tcgen05.mma (kind::f16)
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;          // 16 KiB
constexpr int kBBoxBytes = 64 * BK * 2;       // 8 KiB: 64 columns x 64 K rows
constexpr int kBBytes = BN * BK * 2;          // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
#ifndef EB_EPI_WARPS
#define EB_EPI_WARPS 16
#endif
constexpr int kEpiWarps = EB_EPI_WARPS;             // 8 or 16
constexpr int kEpiGroups = kEpiWarps / 4;           // column groups (each covers all 128 lanes)
constexpr int kEpiCols = BN / kEpiGroups;           // accumulator columns per epilogue warp
static_assert(kEpiCols % 64 == 0, "each epilogue warp takes whole pairs of 32-column chunks");
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kTmemCols = 2 * BN;
constexpr int kMaxCtas = 1024;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 =
// 1), B bf16 (bits 10-12 = 1), A K-major (bit 15 = 0), B N-major (bit 16 = 1), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading byte offset >> 4
// (16-29), stride byte offset >> 4 (32-45), descriptor version 1 (46-47), swizzle mode 2 =
// 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// A (h tile, K-major, 128 rows x 64 K, 128-byte rows swizzled in 8-row / 1024-byte atoms):
// 8-row groups 1024 bytes apart; the K=16 slice k starts 32 k bytes into each row.
__device__ __forceinline__ uint64_t desc_a(uint32_t base, int k)
{
    return smem_desc(base + (uint32_t)k * (UK * 2), 16, 1024);
}

// B (W tile, N-major: four 64-column x 64-K-row boxes of 128-byte rows, 8 KiB apart): 64-column
// blocks are 8192 bytes apart (leading offset), 8-K-row groups 1024 bytes apart (stride
// offset); the K=16 slice k starts 16 k rows = 2048 k bytes in.
__device__ __forceinline__ uint64_t desc_b(uint32_t base, int k)
{
    return smem_desc(base + (uint32_t)k * (UK * 128), kBBoxBytes, 1024);
}

struct Smem {
    static constexpr size_t ring = 0;                                     // 1024-aligned
    static constexpr size_t full = ring + (size_t)kStages * kStageBytes;
    static constexpr size_t empty = full + kStages * 8;
    static constexpr size_t tfull = empty + kStages * 8;
    static constexpr size_t tempty = tfull + 2 * 8;
    static constexpr size_t drain = tempty + 2 * 8;
    static constexpr size_t tmem_base = drain + 8;
    static constexpr size_t abort_flag = tmem_base + 4;
    static constexpr size_t stash = (abort_flag + 4 + 15) & ~(size_t)15;  // 32 B per epilogue thread
    static constexpr size_t total = stash + (size_t)kEpiWarps * 32 * 32;
    static constexpr size_t alloc = total + 1024;                         // alignment slack
};

struct Args {
    const uint8_t *mask;        // [M]
    const int32_t *status;      // [B]
    Partial *partials;          // sampler mode
    float *logits;              // logits mode: [M, V] fp32 out
    int M, K, V, L;
    int MB, NB, KB;
    int g;                      // CTAs per row block (1 when MB > G)
    int G;
    int step;
    float c;                    // log2(e) / T
    float invT;
    RoundKeys keys;
    uint32_t wait_limit;        // mbarrier polls before a wait gives up
    int stall_first;            // diagnostic: the first operand load of each CTA is withheld
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Issues the load of 32 consecutive fp32 accumulator columns of this thread's TMEM lane; the
// registers hold the values only after tc_wait32 on the same array.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Waits for every outstanding tcgen05.ld of the thread.  The array is an in/out operand so
// that no use of the loaded registers moves above the wait.
__device__ __forceinline__ void tc_wait32(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                   "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                   "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Bounded wait that also gives up as soon as another role raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t limit)
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
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    *abort_flag = 1u;
    return false;
}

// Tile iterator shared by the three roles: row blocks mb = mb0, mb0 + mb_step, ...; for each,
// column tiles n = j, j + g, ...
struct Tiles {
    int mb, n, mb_step, j, g, MB, NB;
    __device__ __forceinline__ void begin(const Args &a, int cta)
    {
        if (a.MB <= a.G) {
            mb = cta % a.MB;
            j = cta / a.MB;
            mb_step = a.MB;
        } else {
            mb = cta;
            j = 0;
            mb_step = a.G;
        }
        g = a.g;
        MB = a.MB;
        NB = a.NB;
        n = j;
        if (n >= NB) mb = MB;     // no work (cannot happen: g <= NB)
    }
    __device__ __forceinline__ bool valid() const { return mb < MB; }
    // true when the next tile starts a new row block
    __device__ __forceinline__ bool advance()
    {
        n += g;
        if (n < NB) return false;
        n = j;
        mb += mb_step;
        return true;
    }
};

// ------------------------------------------------------------------ epilogue math

// The 32 accumulator columns r (entries v0 .., v0 a multiple of 32) of this thread's row, as
// four groups of 8 through the streaming kernel's per-group body (each lane owns its row;
// `gumbel` is off for lanes whose row is not masked).
__device__ __forceinline__ void epi_chunk(const uint32_t (&r)[32], int v0, bool on, bool gumbel, const Args &a,
                                          const RowCtx &rc, f32x2 c2, RowState &st, PackedSums &q,
                                          float &nb, f32x2 &nb2, float &K, uint32_t stash)
{
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(r[8 * g + j]);
        const int vg = v0 + 8 * g;
        consume_vals<8, true, false>(x, on && vg < a.V, (uint32_t)vg, a, rc, c2, st, q, nb, nb2, K, gumbel,
                                     stash);
    }
}

__device__ __forceinline__ int partial_flags(const RowState &st, bool ok)
{
    return (ok ? 0 : kPartialTimeout) | ((isnan(st.S) || isnan(st.T2)) ? kPartialNonfinite : 0);
}

// Plain-product mode: the 32 accumulator columns of row r written out as fp32 logits.
__device__ __forceinline__ void store_logits(const uint32_t (&x)[32], int r, int v0, const Args &a)
{
    if (r >= a.M) return;
    float *o = a.logits + (long long)r * a.V + v0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (v0 + j < a.V) o[j] = __uint_as_float(x[j]);
}

// ------------------------------------------------------------------ the kernel

template <bool LOGITS>
__global__ void __launch_bounds__(kThreads, 1)
    k3_unembed(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
               const Args a)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_addr(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Smem::full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Smem::empty);
    uint64_t *tfull = reinterpret_cast<uint64_t *>(smem + Smem::tfull);
    uint64_t *tempty = reinterpret_cast<uint64_t *>(smem + Smem::tempty);
    uint64_t *drain = reinterpret_cast<uint64_t *>(smem + Smem::drain);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::tmem_base);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Smem::abort_flag);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the dependent selection grid may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmap_h);
        prefetch_tmap(&tmap_w);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    Tiles tl;
    tl.begin(a, blockIdx.x);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (; ok && tl.valid();) {
                const int m0 = tl.mb * BM, n0 = tl.n * BN;
                for (int kb = 0; kb < a.KB; ++kb) {
                    const int s = (int)(it % kStages);
                    if (it >= (uint32_t)kStages &&
                        !wait_or_abort(&empty[s], ((it / kStages) & 1u) ^ 1u, abort_flag, a.wait_limit)) {
                        ok = false;
                        break;
                    }
                    if (!(a.stall_first && it == 0)) {
                        const uint32_t st = sbase + (uint32_t)(Smem::ring + (size_t)s * kStageBytes);
                        const uint32_t fb = smem_addr(&full[s]);
                        mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
                        tma_load_2d(st, &tmap_h, kb * BK, m0, fb);
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i)
                            tma_load_2d(st + kABytes + i * kBBoxBytes, &tmap_w, n0 + 64 * i, kb * BK, fb);
                    }
                    ++it;
                }
                tl.advance();
            }
            // every issued copy has landed before the CTA can leave
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
            for (uint32_t q = first; q < it; ++q)
                if (!(a.stall_first && q == 0)) mbar_wait(&full[q % kStages], (q / kStages) & 1u, a.wait_limit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, ti = 0;
            bool ok = true;
            for (; ok && tl.valid();) {
                const uint32_t acc = ti & 1u, use = ti >> 1;
                if (ti >= 2 && !wait_or_abort(&tempty[acc], (use & 1u) ^ 1u, abort_flag, a.wait_limit)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                for (int kb = 0; kb < a.KB; ++kb) {
                    const int s = (int)(it % kStages);
                    if (!wait_or_abort(&full[s], (it / kStages) & 1u, abort_flag, a.wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + (uint32_t)(Smem::ring + (size_t)s * kStageBytes);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k)
                        tc_mma(d, desc_a(sa, k), desc_b(sb, k), kIdesc, (kb | k) != 0 ? 1u : 0u);
                    tc_commit(smem_addr(&empty[s]));
                    ++it;
                }
                if (!ok) break;
                tc_commit(smem_addr(&tfull[acc]));
                ++ti;
                tl.advance();
            }
            // all MMAs issued by this thread are complete before TMEM is released
            tc_commit(smem_addr(drain));
            mbar_wait(drain, 0, a.wait_limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                    // TMEM lane quarter of this warp
        const int hh = (warp - 2) >> 2;            // accumulator column group
        const int rl = 32 * q + lane;              // row within the block
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(hh * kEpiCols);
        const uint32_t stash = sbase + (uint32_t)Smem::stash + (uint32_t)(tid - 64) * 32u;
        uint32_t ti = 0;
        bool ok = true;
        int cur_mb = -1;
        RowState st = empty_state();
        PackedSums qs;
        packed_zero(qs);
        float nb = 0.0f, K = 0.0f;
        f32x2 nb2 = 0ull;
        const f32x2 c2 = pk2(a.c, a.c);
        bool row_on = false, masked = false;
        RowCtx rc{a.c, a.invT, (uint32_t)a.step, 0u, 0u};
        for (; tl.valid();) {
            if (tl.mb != cur_mb) {
                if (!LOGITS && cur_mb >= 0 && row_on) {
                    packed_fold(qs, st);
                    write_partial(&a.partials[((long long)(cur_mb * a.g + tl.j) * kEpiGroups + hh) * BM + rl], st,
                                  partial_flags(st, ok));
                }
                cur_mb = tl.mb;
                const int r = cur_mb * BM + rl;
                row_on = r < a.M;
                if (!LOGITS && row_on) {
                    const int b = r / a.L;
                    row_on = a.status[b] == EB_RUNNING;
                    masked = a.mask[r] != 0;
                    rc.p = (uint32_t)(r - b * a.L);
                    rc.sw = (kStreamGumbel << 24) | (uint32_t)b;
                }
                st = empty_state();
                packed_zero(qs);
                nb = -st.xm * a.c;
                nb2 = pk2(nb, nb);
                K = cand_scale(st.xm, st.best, a.c);
            }
            const uint32_t acc = ti & 1u, use = ti >> 1;
            // one lane waits; the outcome is warp-uniform, as tcgen05.ld needs the whole warp
            int got = 0;
            if (ok && lane == 0) got = wait_or_abort(&tfull[acc], use & 1u, abort_flag, a.wait_limit) ? 1 : 0;
            ok = ok && __shfl_sync(0xFFFFFFFFu, got, 0) != 0;
            tc_fence_after();
            if (ok) {
                const int vbase = tl.n * BN + hh * kEpiCols;
                const uint32_t base = lane_addr + acc * BN;
                // two register buffers: the load of the next chunk is in flight while one runs
                uint32_t ra[32], rb[32];
                tc_ld32(base, ra);
                tc_wait32(ra);
#pragma unroll 1
                for (int ch = 0; ch < kEpiCols / 32; ch += 2) {
                    tc_ld32(base + (uint32_t)(32 * (ch + 1)), rb);
                    const int v0 = vbase + 32 * ch;
                    if (LOGITS) store_logits(ra, cur_mb * BM + rl, v0, a);
                    else epi_chunk(ra, v0, row_on, masked, a, rc, c2, st, qs, nb, nb2, K, stash);
                    tc_wait32(rb);
                    if (ch + 2 < kEpiCols / 32) tc_ld32(base + (uint32_t)(32 * (ch + 2)), ra);
                    if (LOGITS) store_logits(rb, cur_mb * BM + rl, v0 + 32, a);
                    else epi_chunk(rb, v0 + 32, row_on, masked, a, rc, c2, st, qs, nb, nb2, K, stash);
                    if (ch + 2 < kEpiCols / 32) tc_wait32(ra);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&tempty[acc]);
            ++ti;
            tl.advance();
        }
        if (!LOGITS && cur_mb >= 0 && row_on) {
            packed_fold(qs, st);
            write_partial(&a.partials[((long long)(cur_mb * a.g + tl.j) * kEpiGroups + hh) * BM + rl], st,
                          partial_flags(st, ok));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                     : "memory");
    }
}

}  // namespace k3
}  // namespace ebk
