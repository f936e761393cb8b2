// Small-M GEMM (16 <= M <= 64 activation rows) of the 2-bit codebook format
// on the 5th-generation tensor cores (tcgen05), sm_103a.  (The 4-bit format's
// tensor-core kernel is lbq_mma_w4.cu.)
//
// Method (otf-llm 4.0.0, kernel description of its fused INT2 GEMM; SPECTRA
// article, section 4.2 "Batched Tensor Core W4A16 GEMM"): at M >= 16 the
// product Y = X W_hat^T is a real dense contraction, so the packed 2-bit codes
// are dequantised in the kernel to FP16 tiles w_hat = S C[q] + Z (one FP16
// fused multiply-add: one rounding, as the pages' dequantised tiles) and
// multiplied on the tensor cores with FP32 accumulation; the codes cross HBM
// once, in packed form.
//
// GB300 design.  On sm_103a a kind::f16 MMA with M = 128 and K = 16 takes the
// same ~128 clocks for every N from 16 to 256 (measured), so the weights are
// the N = 256 operand and the activations the M = 128 one: each MMA consumes
// 4096 weights, twice what a 128-row weight operand would.
//  * tile = 256 weight rows (64 row blocks of the blob); the work of a call is
//    the sequence of (tile, 256-k chunk) units; a cluster of C CTAs takes a
//    contiguous run of tiles and cuts its units into C contiguous ranges
//    (split-K), so every SM gets the same number of chunks;
//  * tensor memory holds two accumulators of 128 lanes x 256 FP32 columns: a
//    CTA's range spans at most two tiles (taller matrices are cut into slabs
//    of tiles launched one after another), each accumulated in its own D.  The
//    A operand (activations) stays in shared memory: activation stores into
//    tensor memory were measured to stall behind the MMAs' accumulator traffic;
//  * warp roles: 8 dequantising warps (thread = weight row of the tile) load
//    their row's 64 code bytes of each 256-k chunk and the chunk's S and Z
//    straight into registers, one chunk ahead, prefetch their row's line ~8
//    chunks ahead into L2, and turn the codes into the FP16 B stage (256 rows x
//    64 k, the 128-byte swizzled K-major layout the tensor core reads); a copy
//    warp brings each 64-k stage of X (M rows rounded to 8, zero-filled) into
//    the A stage in the same layout (the MMA's 128-row A reads past it into
//    rows whose products land in accumulator lanes that are never read); one
//    thread issues the MMAs (4 per stage) and frees the stages with
//    tcgen05.commit;
//  * codes decode four at a time into a byte-permute selector, so the B stage
//    holds each 16-k block in the order (0,4,8,12,1,5,...); 2 warps (thread =
//    activation row) put the A stage in the same order in place, which leaves
//    the contraction unchanged;
//  * outlier columns (otf-llm's exact FP16 outlier path, in the same kernel as
//    SPECTRA section 4.2's in-kernel outlier fusion) are extra stages of 64
//    columns after a tile's dense chunks: their B stage is the FP16 outlier
//    values of the tile's 256 rows, copied straight into the swizzled B layout
//    by one tensor copy, their A stage x[idx] gathered by the activation warps;
//    the dense A stages carry x~ (the outlier channels zeroed), so every term
//    of y = W_hat x~ + W_out x[idx] lands in the same FP32 accumulator;
//  * partial accumulators of a tile split over several CTAs go through shared
//    memory; each contributing CTA adds one column slice of the tile from all
//    contributors in rank order through distributed shared memory (fixed
//    order: deterministic, no global workspace);
//  * every wait is bounded (2 s of %globaltimer); a timeout records
//    LBQ_ERR_TIMEOUT, makes every other wait of the CTA give up at once, and the
//    CTA drains its copies and tensor-core work, frees its tensor memory and
//    returns.

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kTileRows = 256;                 // weight rows per tile = MMA N
constexpr int kTileRb = kTileRows / 4;         // row blocks per tile
constexpr int kStageK = 64;                    // k per stage (4 MMAs of K = 16)
constexpr int kChunkStages = 4;                // stages per copied chunk (256 k)
constexpr int kChunksPerRec = 1024 / (kStageK * kChunkStages);
constexpr int kDqWarps = 8;                    // dequantising warps: thread = weight row
constexpr int kActWarps = 2;                   // 2-bit: warps ordering the A stage, thread = activation row
constexpr int kIssuers = 1;                    // one thread issues the MMAs
constexpr int kThreads = 32 * (kDqWarps + kActWarps + 1 + kIssuers);   // + X copy warp + MMA warps
// warp roles: a warp's scheduler is warp % 4; the issuing warp's scheduler hosts
// only the two activation warps (the single issuing thread was measured to be
// starved of issue slots next to dequantising warps: ~1000 clocks a stage)
constexpr int kWarpMma = 3;                    // issues the MMAs
constexpr int kWarpAct = 7;                    // activation warps 7 and 11
constexpr int kWarpXCopy = 10;                 // activation copies
// dequantising warps 0, 1, 2, 4, 5, 6, 8, 9 -> index 0..7
__device__ __forceinline__ int dq_index(int warp) { return warp - (warp >= 4) - (warp >= 8); }
constexpr int kNB = 3;                         // B stages (FP16 weights) in shared memory
constexpr int kBStage = kTileRows * 128;       // 32 KB: 256 rows x 64 k x 2 B
constexpr int kNA = 6;                         // A stages in shared memory (X copies run ahead: L2 latency)
constexpr int kNR = 3;                         // raw chunks (codes, S, Z) in shared memory: 2 in flight
constexpr int kAStage = 64 * 128;              // 8 KB: 64 activation rows x 64 k x 2 B
constexpr uint32_t kTmemCols = 512;            // D0 in [0, 256), D1 in [256, 512)
constexpr int kPartStride = 1024 + 16;         // bytes per accumulator row of the partials (padded)
constexpr int kMaxCluster = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// 2-bit record (1536 B): codes (4 rows x 256 B), FP16 S (4 x 32 groups, at 1024), FP16 Z (at 1280)
struct Fmt {
    static constexpr int kRecBytes = 1536;
    static constexpr int kRowCodeBytes = 256;                        // codes of one row in a record
    static constexpr int kChunkRowBytes = kRowCodeBytes / kChunksPerRec;   // 64: one row of a chunk
    static constexpr int kCodeVecs = kChunkRowBytes / 16;            // 16-byte loads per row and chunk
    static constexpr int kMeta0Off = 1024;                           // S
    static constexpr int kMeta1Off = 1280;                           // Z
    static constexpr int kPF = 8;                                    // chunks prefetched into L2 ahead
    static constexpr uint32_t kMagicHi = 0x32334332u;                // "2C32"
    // shared memory: A ring (first: the MMA's A reads run 8 KB past a stage, into
    // the next one or the B ring), B ring, mbarriers, flags
    static constexpr int kA = 0;
    static constexpr int kB = kNA * kAStage;
    // raw chunk: codes of 256 rows x 64 B (each row's four 16-byte parts rotated by
    // row / 2: conflict-free 16-byte reads), then S and Z, 16 B per row
    static constexpr int kRaw = kB + kNB * kBStage;
    static constexpr int kRawS = kTileRows * 64, kRawZ = kRawS + kTileRows * 16;
    static constexpr int kRawStage = kRawZ + kTileRows * 16;         // 24 KB
    static constexpr int kMask = kRaw + kNR * kRawStage;             // outlier-channel bitmask (K bits)
    static constexpr int kBars = kMask + static_cast<int>(lbq::kMaxK / 8);
    static constexpr int kNBars = kNB + 2 * kNA + 2;
    static constexpr int kTotal = kBars + 8 * kNBars + 64 + 4 * (kNB + kNA) + 1024;   // + flags, counters, alignment slack
};

struct Maps {
    CUtensorMap x;
    CUtensorMap out_full;   // outlier records but the last: (column, row, record, row block)
    CUtensorMap out_last;   // the last outlier record of a row block: (column, row, row block)
};

struct MmaArgs {
    const uint8_t* blob;
    const uint8_t* area;    // row block 0
    const __half* x;
    void* y;
    unsigned* err;
    long long ldx, ldy;
    long long N, K;
    long long rb_bytes;
    int n_rb;
    int T;                  // tiles
    int U;                  // dense stages per tile (K / 64)
    int Ud;                 // dense chunks per tile (256 k each; the last may be short)
    int OS;                 // outlier stages per tile (64 columns each)
    int Ut;                 // stages per tile: U dense, then OS outlier stages
    int n_out;              // outlier columns
    int OT;                 // outlier records per row block
    int recs;               // dense records per row block
    int cols_last;          // columns of the last outlier record (a multiple of 8)
    const int32_t* idx;     // outlier channel indices (device, in the blob)
    int C;                  // CTAs per cluster
    int G;                  // clusters
    int M;                  // activation rows
    int Mr;                 // rows of an X copy: M rounded up to 8
    int y_f32;
    long long N_hdr;        // rows of the whole blob (a slab's launch checks the header against it)
    uint32_t lut_lo, lut_hi;   // 2-bit codebook as FP16 byte tables
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}


__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the limit.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// UMMA shared-memory descriptor of a K-major operand in the 128-byte swizzled
// layout: 8-row atoms of 8 x 128 bytes, 1024 bytes apart (SBO); version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;                 // LBO (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // SBO
    d |= 1ull << 46;                                      // descriptor version for tcgen05
    d |= 2ull << 61;                                      // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: A, B FP16 (K-major), D FP32, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4)                                  // D format: F32
           | (0u << 7) | (0u << 10)                   // A, B format: F16
           | (0u << 15) | (0u << 16)                  // A, B K-major
           | (static_cast<uint32_t>(n >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// 16-byte copy global -> shared that completes asynchronously (zero fill when
// src_bytes is 0; the source is then not read)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t u4w(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Word v of a row's 2-bit codes (16 codes, byte i = codes of k = 4i..4i+3) as
// 16 dequantised FP16 weights S C[q] + Z (one rounding), in the stage order
// slot p <-> k = 4 (p % 4) + p / 4: out[2 sh] = (w_{sh}, w_{4+sh}),
// out[2 sh + 1] = (w_{8+sh}, w_{12+sh}).
__device__ __forceinline__ void w2_word(uint32_t w, uint32_t S2, uint32_t Z2, uint32_t lut_lo, uint32_t lut_hi,
                                        uint32_t (&out)[8]) {
#pragma unroll
    for (int sh = 0; sh < 4; ++sh) {
        const uint32_t t = (w >> (2 * sh)) & 0x03030303u;
        const uint32_t sel = t * 0x11u + 0x40404040u;   // nibbles (c, c + 4) per code
        out[2 * sh] = hfma2(prmt(lut_lo, lut_hi, sel), S2, Z2);
        out[2 * sh + 1] = hfma2(prmt(lut_lo, lut_hi, sel >> 16), S2, Z2);
    }
}

// 16 activations of one 16-k block (natural pairs n[0..7]) in the 2-bit stage
// order: pairs (0,4) (8,12) (1,5) (9,13) (2,6) (10,14) (3,7) (11,15).
__device__ __forceinline__ void w2_order(const uint32_t (&n)[8], uint32_t (&o)[8]) {
    o[0] = prmt(n[0], n[2], 0x5410u);
    o[1] = prmt(n[4], n[6], 0x5410u);
    o[2] = prmt(n[0], n[2], 0x7632u);
    o[3] = prmt(n[4], n[6], 0x7632u);
    o[4] = prmt(n[1], n[3], 0x5410u);
    o[5] = prmt(n[5], n[7], 0x5410u);
    o[6] = prmt(n[1], n[3], 0x7632u);
    o[7] = prmt(n[5], n[7], 0x7632u);
}

}  // namespace

namespace {

__global__ void __launch_bounds__(kThreads, 1)
    lbq_w2_mma_kernel(const __grid_constant__ MmaArgs a, const __grid_constant__ Maps maps) {
    using F = Fmt;
    constexpr uint32_t kIdesc = idesc_f16(128, kTileRows);
    static_assert(128 * kPartStride <= F::kBars, "the partial accumulators reuse the stage rings");
    static_assert(F::kTotal <= 232448, "shared memory of one CTA");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    // mbarriers (one arrival each: a tensor-core commit or a copy's issuing thread):
    // B stage free [kNB], X copied [kNA], A stage free [kNA], accumulators done,
    // outlier copy landed
    const uint32_t bempty = sb + F::kBars, xfull = bempty + 8 * kNB, aempty = xfull + 8 * kNA,
                   dfull = aempty + 8 * kNA, ocopy = dfull + 8;
    uint32_t* flags = reinterpret_cast<uint32_t*>(smem + F::kBars + 8 * F::kNBars);
    volatile uint32_t* abort_flag = flags + 1;
    // per ring slot, the arrivals of the warps that fill it (dequantising warps for a
    // B slot, activation warps for an A slot), counted over the slot's rounds: round
    // r of a slot is ready at (r + 1) x warps (no warp reaches the next round before
    // the MMAs of this one have freed the slot).  The issuing thread polls these with
    // plain acquire loads: an mbarrier wait right after its commits was measured to
    // hold it until the tensor core had drained (the MMAs ran ~30 % of the time)
    const uint32_t bready = smem_u32(flags + 16), aready = bready + 4 * kNB;
    volatile int* xissued = reinterpret_cast<volatile int*>(flags + 4);  // X stages whose copies were issued

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = a.C, U = a.U, Ut = a.Ut;
    const int cl = static_cast<int>(blockIdx.x) / C, rank = static_cast<int>(blockIdx.x) % C;
    int t0, t1;
    lbq::cluster_tiles(a.T, a.G, cl, &t0, &t1);
    const int units = (t1 - t0) * Ut;
    int lu0, lu1;
    lbq::rank_range(units, C, rank, &lu0, &lu1);
    // this CTA's stages: units [u0, u1) of the cluster, unit u = stage u % Ut of tile
    // t0 + u / Ut (stage c < U: k in [64 c, 64 c + 64); c >= U: outlier columns
    // [64 (c - U), 64 (c - U) + 64))
    const int u0 = lu0, u1 = lu1;
    const int nst = u1 - u0;
    const int first_tile = t0 + (nst > 0 ? u0 / Ut : 0);
    const int nbands = nst > 0 ? (u1 - 1) / Ut - u0 / Ut + 1 : 0;   // tiles touched (<= 2)

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(flags)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    uint32_t* omask = reinterpret_cast<uint32_t*>(smem + F::kMask);   // bit k: channel k is an outlier
    if (a.n_out > 0)
        for (int i = tid; i < static_cast<int>((a.K + 31) / 32); i += kThreads) omask[i] = 0u;
    if (tid == 32) {
        for (int i = 0; i < F::kNBars; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bempty + 8 * i) : "memory");
        *abort_flag = 0;
        for (int i = 0; i < kNB + kNA; ++i) flags[16 + i] = 0u;
        *xissued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = flags[0];
    for (int i = tid; i < a.n_out; i += kThreads) {
        const int k = a.idx[i];
        if (k >= 0 && k < a.K)
            atomicOr(&omask[k >> 5], 1u << (k & 31));
        else
            atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_OUTLIER_IDX));   // corrupted blob: never index outside x
    }
    if (warp < 4) {
        // clear both accumulators (every MMA accumulates): warp w zeroes lane quarter w
#pragma unroll 1
        for (int c0 = 0; c0 < static_cast<int>(kTmemCols); c0 += 32)
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, "
                "%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(
                    tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(c0)),
                "r"(0u)
                : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // bounded wait that gives up at once after any thread of the CTA gave up
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t w0 = global_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (*abort_flag) return false;
            if (global_ns() - w0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
                return false;
            }
        }
        return true;
    };
    auto count_up = [&](uint32_t counter) {
        asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" ::"r"(counter) : "memory");
    };
    auto commit = [&](uint32_t bar) {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    };
    // lane 0 waits for the warp; the others follow after __syncwarp
    auto warp_wait = [&](uint32_t bar, uint32_t parity, bool cond) -> bool {
        bool ok = true;
        if (lane == 0 && cond) ok = wait(bar, parity);
        __syncwarp();
        return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };

    if (warp == kWarpXCopy) {
        // ------------------------------------------------------------------ activation copies
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");   // X may be written by the previous kernel
            int i = 0, c = u0 % Ut;
            for (; i < nst; ++i, c = c + 1 == Ut ? 0 : c + 1) {
                const int as = i % kNA;
                if (i >= kNA && !wait(aempty + 8 * as, ((i - kNA) / kNA) & 1)) break;
                if (c < U) {
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(xfull + 8 * as),
                                 "r"(static_cast<uint32_t>(a.Mr * 128))
                                 : "memory");
                    asm volatile(
                        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                        " [%0], [%1, {%2, %3}], [%4];" ::"r"(sb + F::kA + as * kAStage),
                        "l"(&maps.x), "r"(c * kStageK), "r"(0), "r"(xfull + 8 * as)
                        : "memory");
                } else {
                    // outlier stage: the activation warps gather its A stage; the slot is free
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(xfull + 8 * as) : "memory");
                }
            }
            *xissued = i;
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ tensor-core issue
        // one thread, stages in order (D sums them in a fixed order); its waits poll
        // the ready counters, bounded like every other wait
        auto poll = [&](uint32_t counter, uint32_t target) -> bool {
            if (ld_acquire_u32(counter) >= target) return true;
            const uint64_t w0 = global_ns();
            while (ld_acquire_u32(counter) < target) {
                if (*abort_flag) return false;
                if (global_ns() - w0 > kWaitLimitNs) {
                    *abort_flag = 1;
                    atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
                    return false;
                }
            }
            return true;
        };
        if (lane == 0) {
            int i = 0, as = 0, bs = 0;          // stage, its A and B slots
            uint32_t ra = kActWarps, rb = kDqWarps;   // arrivals that make slots as, bs ready
            for (int c = u0 % Ut, t = first_tile; i < nst; ++i, c = c + 1 == Ut ? 0 : c + 1) {
                if (c == 0 && i > 0) ++t;
                const uint32_t d = tmem + (t == first_tile ? 0u : static_cast<uint32_t>(kTileRows));
                {
                    bool ok = poll(aready + 4 * as, ra) && poll(bready + 4 * bs, rb);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    if (ok) {
                        const uint64_t da = smem_desc_sw128(sb + F::kA + as * kAStage),
                                       db = smem_desc_sw128(sb + F::kB + bs * kBStage);
#pragma unroll
                        for (int ks = 0; ks < kStageK / 16; ++ks)   // +32 bytes of K per MMA
                            asm volatile(
                                "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, 1, 1;\n\t"
                                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                                "l"(da + 2 * ks), "l"(db + 2 * ks), "r"(kIdesc)
                                : "memory");
                    }
                    // always commit, so that every wait on these stages completes
                    commit(bempty + 8 * bs);
                    commit(aempty + 8 * as);
                    if (++as == kNA) {
                        as = 0;
                        ra += kActWarps;
                    }
                    if (++bs == kNB) {
                        bs = 0;
                        rb += kDqWarps;
                    }
                }
            }
            if (nst > 0) commit(dfull);   // tracks every tensor-core operation of the CTA
        }
        __syncwarp();
    } else if ((warp & 3) == 3) {
        // ------------------------------------------------------------------ A stages: order, mask, gather
        // dense stage: the copied X in the codes' decode order, outlier channels
        // zeroed (x~); outlier stage: x[idx_j] of its 64 outlier columns, in order
        {
            const int m = 32 * (warp == kWarpAct ? 0 : 1) + lane;   // A row: 128 bytes at its swizzled place
            const uint32_t arow = static_cast<uint32_t>((m >> 3) * 1024 + (m & 7) * 128), asw = static_cast<uint32_t>(m & 7);
            for (int i = 0, c = u0 % Ut; i < nst; ++i, c = c + 1 == Ut ? 0 : c + 1) {
                const int as = i % kNA;
                const bool ok = warp_wait(xfull + 8 * as, (i / kNA) & 1, true);
                if (ok && !*abort_flag) {
                    const uint32_t row = sb + F::kA + as * kAStage + arow;
                    uint32_t w[32];
                    if (c >= U) {
                        // outlier stage: x[idx_j] of its 64 outlier columns, in order.  Lane l
                        // gathers columns l and 32 + l of 16-row batches - activation warp w
                        // takes rows 16 w .. 16 w + 15 and 32 + 16 w .. 32 + 16 w + 15 - with
                        // every load of a batch in flight (rows past M and invalid channels
                        // give 0), and stores them in place, 2 bytes each, at their swizzled
                        // positions
                        const int j0 = kStageK * (c - U);   // first outlier column
                        const int ja = j0 + lane, jb = j0 + 32 + lane;
                        const int ka = ja < a.n_out ? __ldg(a.idx + ja) : -1;
                        const int kb = jb < a.n_out ? __ldg(a.idx + jb) : -1;
                        const bool oka = ka >= 0 && ka < a.K, okb = kb >= 0 && kb < a.K;
                        const unsigned short* xs = reinterpret_cast<const unsigned short*>(a.x);
                        const uint32_t abase = sb + F::kA + as * kAStage;
                        const uint32_t ca = static_cast<uint32_t>(lane >> 3), off = static_cast<uint32_t>((lane & 7) * 2);
                        auto gather_rows = [&](int mb) {
                            unsigned short va[16], vb[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int mm = mb + e;
                                const unsigned short* xr = xs + (mm < a.M ? mm : 0) * a.ldx;
                                va[e] = __ldg(xr + (oka ? ka : 0));
                                vb[e] = __ldg(xr + (okb ? kb : 0));
                            }
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int mm = mb + e;
                                if (mm < a.Mr) {
                                    const uint32_t rw = abase + static_cast<uint32_t>((mm >> 3) * 1024 + (mm & 7) * 128);
                                    const uint32_t sw7 = static_cast<uint32_t>(mm & 7);
                                    const unsigned short lo = mm < a.M && oka ? va[e] : 0, hi = mm < a.M && okb ? vb[e] : 0;
                                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(rw + ((ca ^ sw7) << 4) + off), "h"(lo) : "memory");
                                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(rw + (((ca + 4u) ^ sw7) << 4) + off), "h"(hi)
                                                 : "memory");
                                }
                            }
                        };
#pragma unroll 1
                        for (int mb = m - lane == 0 ? 0 : 16; mb < a.Mr; mb += 32) gather_rows(mb);   // this warp's batches
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // read by the tensor core
                    } else if (m < a.Mr) {
                        const int s = c;   // k in [64 s, 64 s + 64)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 v = lds128(row + ((j ^ asw) << 4));
                            w[4 * j] = v.x;
                            w[4 * j + 1] = v.y;
                            w[4 * j + 2] = v.z;
                            w[4 * j + 3] = v.w;
                        }
                        if (a.n_out > 0) {
                            const uint32_t mk[2] = {omask[2 * s], omask[2 * s + 1]};
                            if (mk[0] | mk[1]) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    const uint32_t bits = (mk[e >> 4] >> (2 * (e & 15))) & 3u;
                                    w[e] &= ((bits & 1u) ? 0xFFFF0000u : 0xFFFFFFFFu) & ((bits & 2u) ? 0x0000FFFFu : 0xFFFFFFFFu);
                                }
                            }
                        }
#pragma unroll
                        for (int blk = 0; blk < 4; ++blk) {
                            uint32_t nat[8], o[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) nat[e] = w[8 * blk + e];
                            w2_order(nat, o);
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[8 * blk + e] = o[e];
                        }
                    }
                    if (c < U && m < a.Mr) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            sts128(row + ((j ^ asw) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // read by the tensor core
                    }
                }
                __syncwarp();
                if (lane == 0) count_up(aready + 4 * as);
            }
        }
    } else {
        // ------------------------------------------------------------------ dequantisation -> B stages
        // thread = weight row n of the tile (row block n / 4, row n % 4); its codes and
        // metadata come straight from global memory into registers, one chunk ahead
        const int dw = dq_index(warp), n = 32 * dw + lane, rbl = n >> 2, r = n & 3;
        const uint32_t brow = static_cast<uint32_t>((n >> 3) * 1024 + (n & 7) * 128);   // row n of a B stage
        const uint32_t sw = static_cast<uint32_t>(n & 7);                               // its 128-byte swizzle
        const uint32_t lut_lo = a.lut_lo, lut_hi = a.lut_hi;
        constexpr int CV = F::kCodeVecs;
        // The stages are consumed in groups: a group is the CTA's run of stages inside
        // one chunk (4 dense stages = 256 k, or 4 outlier stages = 256 columns).  Group
        // starting at unit g ends where the chunk does (or at u1):
        auto group_end = [&](int g) -> int {
            const int c = g % Ut;
            const int ce = c < U ? min(c - c % kChunkStages + kChunkStages, U)
                                 : U + min(c - U - (c - U) % kChunkStages + kChunkStages, Ut - U);
            return min(g + (ce - c), u1);
        };
        // copies of the dense group at unit g into raw slot `slot`: of the chunk, the
        // codes of the group's stages (16 B a row and stage; 4 lanes a row: whole 32-byte
        // sectors) and the chunk's S and Z (lane = row)
        auto copy_group = [&](int g, int slot_i) {
            const int t = t0 + g / Ut, c = g % Ut;
            if (c >= U) return;
            const int p0 = c % kChunkStages, p1 = p0 + (group_end(g) - g);   // parts (stages) to copy
            const uint32_t slot = sb + F::kRaw + slot_i * F::kRawStage;
            const int cc = (c / kChunkStages) % kChunksPerRec;
            const long long rec_off = static_cast<long long>(c / (kChunkStages * kChunksPerRec)) * F::kRecBytes;
#pragma unroll
            for (int v = 0; v < F::kCodeVecs; ++v) {
                const int rw = 8 * v + (lane >> 2), part = lane & 3, nr = 32 * dw + rw;
                const int rb = t * kTileRb + (nr >> 2);
                if (rb < a.n_rb && part >= p0 && part < p1)
                    cp_async16(slot + nr * 64 + (((part + (rw >> 1)) & 3) << 4),
                               a.area + static_cast<long long>(rb) * a.rb_bytes + rec_off +
                                   (nr & 3) * F::kRowCodeBytes + cc * F::kChunkRowBytes + 16 * part,
                               16u);
            }
            const int rb = t * kTileRb + rbl;
            const bool in = rb < a.n_rb;   // rows past the matrix: zero S and Z, so zero weights
            const uint8_t* rec = a.area + (in ? static_cast<long long>(rb) * a.rb_bytes + rec_off + r * 64 + 16 * cc : 0);
            cp_async16(slot + F::kRawS + 16 * n, rec + (in ? F::kMeta0Off : 0), in ? 16u : 0u);
            cp_async16(slot + F::kRawZ + 16 * n, rec + (in ? F::kMeta1Off : 0), in ? 16u : 0u);
        };
        // row n's FP16 outlier values of outlier stage os (64 columns) and where they sit
        auto out_row = [&](int t, int os) -> const uint8_t* {
            const int rb = t * kTileRb + rbl, j0 = kStageK * os, o = j0 / lbq::kOutlierCols;
            if (rb >= a.n_rb) return nullptr;
            const int cols = o + 1 < a.OT ? lbq::kOutlierCols : a.cols_last;
            return a.area + static_cast<long long>(rb) * a.rb_bytes + static_cast<long long>(a.recs) * F::kRecBytes +
                   static_cast<long long>(o) * (lbq::kOutlierCols * lbq::kRowsPerBlock * 2) + r * cols * 2 +
                   (j0 % lbq::kOutlierCols) * 2;
        };
        // L2 prefetch of the group at unit g: row n's lines
        auto prefetch_group = [&](int g) {
            const int t = t0 + g / Ut, c = g % Ut, rb = t * kTileRb + rbl;
            if (rb >= a.n_rb) return;
            if (c >= U) {
                for (int e = g; e < group_end(g); ++e) {
                    const uint8_t* p = out_row(t, c - U + (e - g));
                    if (p) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
                }
                return;
            }
            const int cc = (c / kChunkStages) % kChunksPerRec;
            const uint8_t* rec = a.area + static_cast<long long>(rb) * a.rb_bytes +
                                 static_cast<long long>(c / (kChunkStages * kChunksPerRec)) * F::kRecBytes;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + r * F::kRowCodeBytes + cc * F::kChunkRowBytes));
            if (r == 0 && (cc == 0 || g == u0)) {
                // the row block's S and Z lines of the record (512 B)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + F::kMeta0Off));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + F::kMeta0Off + 128));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + F::kMeta0Off + 256));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + F::kMeta0Off + 384));
            }
        };
        int gc = u0;   // next group to copy
        for (int j = 0; j < kNR - 1; ++j) {
            if (gc < u1) {
                copy_group(gc, j);
                gc = group_end(gc);
            }
            cp_async_commit();
        }
        int gp = u0;   // next group to prefetch into L2
        for (int j = 0; j < F::kPF && gp < u1; ++j) {
            if (j > 0) prefetch_group(gp);
            gp = group_end(gp);
        }
        int is = 0;         // stage index
        int n_copies = 0;   // outlier copies issued (warp 0, lane 0)
        for (int g = u0, j = 0; g < u1; ++j) {
            const int ge = group_end(g), t = t0 + g / Ut, c0 = g % Ut;
            __syncwarp();   // every lane has read the slot that the next copies refill
            if (gc < u1) {
                copy_group(gc, (j + kNR - 1) % kNR);
                gc = group_end(gc);
            }
            cp_async_commit();
            if (gp < u1) {
                prefetch_group(gp);
                gp = group_end(gp);
            }
            cp_async_wait<kNR - 1>();   // this lane's copies of group j have landed
            __syncwarp();               // and every lane's
            uint4 q[CV], m0, m1;
            {
                const uint32_t slot = sb + F::kRaw + (j % kNR) * F::kRawStage;
#pragma unroll
                for (int v = 0; v < CV; ++v) q[v] = lds128(slot + n * 64 + (((v + (n >> 1)) & 3) << 4));
                m0 = lds128(slot + F::kRawS + 16 * n);
                m1 = lds128(slot + F::kRawZ + 16 * n);
            }
            const int jj0 = c0 < U ? c0 % kChunkStages : (c0 - U) % kChunkStages;   // first stage in the chunk
#pragma unroll
            for (int jj = 0; jj < kChunkStages; ++jj) {
                if (jj < jj0 || jj >= jj0 + (ge - g)) continue;
                const int bs = is % kNB;
                const uint32_t bst = sb + F::kB + bs * kBStage + brow;
                if (c0 >= U) {
                    const bool ok = warp_wait(bempty + 8 * bs, ((is - kNB) / kNB) & 1, is >= kNB);
                    // outlier stage: the tile's 256 rows x 64 FP16 outlier values go straight
                    // into the B stage (the copy writes the swizzled layout); warp 0 issues the
                    // copy and waits for it to land before its arrival, so that no copy is in
                    // flight when the CTA ends, whatever happened
                    if (lane == 0 && warp == 0 && ok && !*abort_flag) {
                        const int j0 = kStageK * (c0 - U - jj0 + jj);
                        const int o = j0 / lbq::kOutlierCols, col = j0 % lbq::kOutlierCols;
                        const uint32_t dst = sb + F::kB + bs * kBStage;
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(ocopy), "r"(kBStage)
                                     : "memory");
                        if (o + 1 < a.OT)
                            asm volatile(
                                "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
                                "l"(&maps.out_full), "r"(col), "r"(0), "r"(o), "r"(t * kTileRb), "r"(ocopy)
                                : "memory");
                        else
                            asm volatile(
                                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
                                "l"(&maps.out_last), "r"(col), "r"(0), "r"(t * kTileRb), "r"(ocopy)
                                : "memory");
                        if (!mbar_wait(ocopy, n_copies & 1, kWaitLimitNs)) {
                            *abort_flag = 1;
                            atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
                        }
                        ++n_copies;
                    }
                    __syncwarp();
                    if (lane == 0) count_up(bready + 4 * bs);
                    ++is;
                    continue;
                }
                // dense stage: decode first (it needs no slot), then wait for the slot and store
                uint32_t o[4][8];
                {
                    const uint4 qs = q[jj];
                    const uint32_t Sw = u4w(m0, jj), Zw = u4w(m1, jj);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int qg = v >> 1;   // 32-k quantisation group of the stage
                        const uint32_t S2 = ((Sw >> (16 * qg)) & 0xFFFFu) * 0x00010001u;
                        const uint32_t Z2 = ((Zw >> (16 * qg)) & 0xFFFFu) * 0x00010001u;
                        w2_word(u4w(qs, v), S2, Z2, lut_lo, lut_hi, o[v]);
                    }
                }
                const bool ok = warp_wait(bempty + 8 * bs, ((is - kNB) / kNB) & 1, is >= kNB);
                if (ok && !*abort_flag) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        sts128(bst + (((2 * v) ^ sw) << 4), o[v][0], o[v][1], o[v][2], o[v][3]);
                        sts128(bst + (((2 * v + 1) ^ sw) << 4), o[v][4], o[v][5], o[v][6], o[v][7]);
                    }
                }
                // the B stage is read by the tensor core (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) count_up(bready + 4 * bs);
                ++is;
            }
            g = ge;
        }
        cp_async_wait<0>();   // no copy outlives the loop, whatever happened
    }

    // ---------------------------------------------------------------------- epilogue
    // the accumulator is complete once the last commit has arrived
    const bool got = nst == 0 || mbar_wait(dfull, 0, kWaitLimitNs);
    if (!got && tid == 0) atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
    __syncthreads();
    const bool bad = *abort_flag != 0 || !got;
    // after an abort the last code copies issued may still be in flight: wait for them
    if (bad && tid == 32 * kWarpXCopy) {
        const int ix = *xissued;
        for (int i = ix > kNA ? ix - kNA : 0; i < ix; ++i)
            mbar_wait(xfull + 8 * (i % kNA), (i / kNA) & 1, kWaitLimitNs / 64);
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // contributors of tile t: the ranks whose ranges hold its first and last stage
    auto contributors = [&](int t, int* rlo, int* rhi) {
        *rlo = lbq::rank_of(units, C, (t - t0) * Ut);
        *rhi = lbq::rank_of(units, C, (t - t0 + 1) * Ut - 1);
    };
    auto store_y = [&](int m, long long n, float v) {
        if (a.y_f32)
            reinterpret_cast<float*>(a.y)[m * a.ldy + n] = v;
        else
            reinterpret_cast<__half*>(a.y)[m * a.ldy + n] = __float2half_rn(v);
    };
    // D -> shared memory: warps 0, 1, 4, 5 read lane quarter warp % 4 (activation
    // rows 32 (warp % 4) ..) and columns 128 (warp / 4) .. + 127 of each accumulator
    // into row 64 b + m of the partials (padded rows: conflict-free 16-byte stores)
    if (warp < kDqWarps && (warp & 3) < 2 && 32 * (warp & 3) < a.M && !bad) {
        const int q = warp & 3, h = warp >> 2;
        const int m = 32 * q + lane;
        for (int b = 0; b < nbands; ++b) {
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                const int col0 = 128 * h + 32 * cc;
                uint32_t v[32];
                __syncwarp();   // tcgen05.ld is warp-collective
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                    "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
                    "[%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                      "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                      "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                      "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                      "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(kTileRows * b + col0)));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (m < a.M) {
                    const uint32_t p = sb + static_cast<uint32_t>((64 * b + m) * kPartStride + col0 * 4);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) sts128(p + 4 * j, v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
        }
    }
    // every CTA's partials are in place; a tile is summed over its contributors in
    // rank order, each contributor taking one column slice, and written along the
    // columns (4 columns a thread, consecutive threads consecutive columns)
    if (C > 1)
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    else
        __syncthreads();
    if (!bad) {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the previous kernel is done with y
        for (int b = 0; b < nbands; ++b) {
            const int t = first_tile + b;
            int rlo, rhi;
            contributors(t, &rlo, &rhi);
            const int nc = rhi - rlo + 1, ci = rank - rlo;
            const int c0 = 4 * ((64 * ci) / nc), c1 = 4 * ((64 * (ci + 1)) / nc);
            const int w4 = (c1 - c0) / 4;
            if (w4 <= 0) continue;
            // the contributors' band of this tile: 0, except for the first contributor
            // when its range starts in the tile before
            const int bp_lo = t0 + (units * rlo / C) / Ut < t ? 1 : 0;
            const int ne = a.M * w4;
            for (int e0 = tid; e0 < ne; e0 += 2 * kThreads) {
                // two elements a thread, every load of both in flight, then the sums in rank order
                float4 pv[2][kMaxCluster];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = e0 + h * kThreads;
                    if (e >= ne) break;
                    const int m = e / w4, cq = e - m * w4;
#pragma unroll
                    for (int k = 0; k < kMaxCluster; ++k) {
                        if (k >= nc) break;
                        const int bp = k == 0 ? bp_lo : 0;
                        const uint32_t local =
                            sb + static_cast<uint32_t>((64 * bp + m) * kPartStride + (c0 + 4 * cq) * 4);
                        if (C > 1) {
                            uint32_t remote;
                            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rlo + k));
                            asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(pv[h][k].x), "=f"(pv[h][k].y), "=f"(pv[h][k].z), "=f"(pv[h][k].w)
                                         : "r"(remote));
                        } else {
                            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(pv[h][k].x), "=f"(pv[h][k].y), "=f"(pv[h][k].z), "=f"(pv[h][k].w)
                                         : "r"(local));
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e = e0 + h * kThreads;
                    if (e >= ne) break;
                    const int m = e / w4, cq = e - m * w4;
                    float4 sum = pv[h][0];
#pragma unroll
                    for (int k = 1; k < kMaxCluster; ++k) {
                        if (k >= nc) break;
                        sum.x += pv[h][k].x;
                        sum.y += pv[h][k].y;
                        sum.z += pv[h][k].z;
                        sum.w += pv[h][k].w;
                    }
                    const long long n = static_cast<long long>(t) * kTileRows + c0 + 4 * cq;
                    if (n < a.N) store_y(m, n, sum.x);
                    if (n + 1 < a.N) store_y(m, n + 1, sum.y);
                    if (n + 2 < a.N) store_y(m, n + 2, sum.z);
                    if (n + 3 < a.N) store_y(m, n + 3, sum.w);
                }
            }
        }
    }
    // no CTA leaves while another may still read its shared memory
    if (C > 1)
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (blockIdx.x == 0 && tid == 0) {
        const uint4* hp = reinterpret_cast<const uint4*>(a.blob);
        const uint4 h0 = hp[0], h1 = hp[1], h2 = hp[2];
        const long long n_hdr = (static_cast<long long>(h1.y) << 32) | h1.x;
        const long long k_hdr = (static_cast<long long>(h1.w) << 32) | h1.z;
        if (h0.x != 0x5751424Cu || h0.y != F::kMagicHi || h0.z != LBQ_FORMAT_VERSION_NUM || n_hdr != a.N_hdr ||
            k_hdr != a.K || static_cast<int>(h2.x) != a.n_out)
            atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_FORMAT));
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

const void* kernel_fn() { return reinterpret_cast<const void*>(&lbq_w2_mma_kernel); }

// Clusters of each size that fit the device at once (0: that size cannot be
// launched), per device and kind, looked up once.
constexpr int kMaxDev = 64;
std::mutex g_plan_mu;
int g_active[kMaxDev][kMaxCluster + 1];
bool g_active_init[kMaxDev];

lbq_status active_clusters(int max_smem, const int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return LBQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (!g_active_init[dev]) {
        const void* fn = kernel_fn();
        const int smem = Fmt::kTotal;
        if (smem > max_smem) return LBQ_ERR_SHAPE;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            (void)cudaGetLastError();
            return LBQ_ERR_CUDA;
        }
        for (int c = 1; c <= kMaxCluster; ++c) {
            cudaLaunchConfig_t cfg;
            std::memset(&cfg, 0, sizeof(cfg));
            cfg.gridDim = dim3(static_cast<unsigned>(c));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = static_cast<size_t>(smem);
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(c);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();
                n = 0;
            }
            g_active[dev][c] = n;
        }
        g_active_init[dev] = true;
    }
    *out = g_active[dev];
    return LBQ_OK;
}

}  // namespace

namespace lbq {

// Work plan of the tensor-core kernel over T tiles of Ut stages: the cluster
// size C and cluster count G that give the fewest chunks to the busiest CTA,
// with every CTA's range spanning at most as many tiles as the accumulator has
// lane bands.  False when no cluster size fits.
bool mma_plan(int T, int Ut, int bands, const int* active, int* C_out, int* G_out, int* load_out) {
    // the split is evaluated in 32-bit arithmetic on the device
    if (T < 1 || Ut < 1 || T > 32768 || static_cast<long long>(T) * Ut * kMaxCluster >= (1ll << 31)) return false;
    int bestC = 0, bestG = 0;
    long long best = -1;
    for (int c = 1; c <= kMaxCluster; ++c) {
        int g = active[c];
        if (g <= 0) continue;
        if (g > T) g = T;
        long long load = 0;
        bool fits = true;
        for (int cl = 0; cl < g && fits; ++cl) {
            int t0, t1;
            cluster_tiles(T, g, cl, &t0, &t1);
            const int units = (t1 - t0) * Ut;
            for (int r = 0; r < c; ++r) {
                int u0, u1;
                rank_range(units, c, r, &u0, &u1);
                if (u1 - u0 > load) load = u1 - u0;
                if (u1 > u0 && (u1 - 1) / Ut - u0 / Ut + 1 > bands) fits = false;
            }
        }
        // fewer chunks per CTA wins; on a tie the smaller cluster (less reduction)
        if (fits && (best < 0 || load < best)) {
            best = load;
            bestC = c;
            bestG = g;
        }
    }
    if (best < 0) return false;
    *C_out = bestC;
    *G_out = bestG;
    *load_out = static_cast<int>(best);
    return true;
}

// Launch the tensor-core GEMM for one problem (16 <= M <= 64, any number of
// outlier columns): one launch per slab of tiles, each slab small enough that
// every CTA's range spans at most two tiles.  With `launches` set, only counts
// the launches.  Returns LBQ_ERR_SHAPE when the problem does not fit the kernel.
lbq_status launch_w2_mma(const void* packed, int64_t N, int64_t K, int32_t n_out, int M, const void* x, int64_t ldx,
                         void* y, int64_t ldy, bool y_f32, unsigned* err_word, int max_smem, void* stream,
                         uint32_t flags, int* launches) {
    if (M < 16 || M > 64) return LBQ_ERR_SHAPE;
    lbq_layout L;
    lbq_status st = lbq_blob_layout(LBQ_KIND_W2CB, N, K, n_out, &L);
    if (st != LBQ_OK) return st;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return LBQ_ERR_CUDA;
    const int* active = nullptr;
    st = active_clusters(max_smem, &active);
    if (st != LBQ_OK) return st;
    const int T = static_cast<int>((N + kTileRows - 1) / kTileRows);
    // chunk units of a tile: the dense chunks (256 k each), then the outlier chunks
    // (256 outlier columns each, in 64-column stages)
    const int U = static_cast<int>(K / kStageK), Ud = (U + kChunkStages - 1) / kChunkStages;
    const int OS = (n_out + kStageK - 1) / kStageK, Ut = U + OS;
    const int OT = static_cast<int>(L.outlier_records);
    const int cols_last = n_out > 0 ? (n_out + lbq::kOutlierColAlign - 1) / lbq::kOutlierColAlign *
                                              lbq::kOutlierColAlign - (OT - 1) * lbq::kOutlierCols
                                    : 0;
    int slab = T, C = 0, G = 0, load = 0;
    while (slab > 1 && !mma_plan(slab, Ut, 2, active, &C, &G, &load)) slab = (slab + 1) / 2;
    if (!mma_plan(slab, Ut, 2, active, &C, &G, &load)) return LBQ_ERR_SHAPE;
    if (launches) {
        *launches += (T + slab - 1) / slab;
        return LBQ_OK;
    }
    // 2-bit codebook as FP16 byte tables for PRMT (otf-llm section 2, rounded once)
    uint32_t lut_lo = 0, lut_hi = 0;
    const double cb[4] = {-1.52, -0.45, 0.45, 1.52};
    for (int c = 0; c < 4; ++c) {
        const uint16_t h = lbq::host_f64_to_f16(cb[c]);
        lut_lo |= uint32_t(h & 0xFF) << (8 * c);
        lut_hi |= uint32_t(h >> 8) << (8 * c);
    }
    const void* fn = kernel_fn();
    const int smem = Fmt::kTotal;
    uint8_t* b = static_cast<uint8_t*>(const_cast<void*>(packed));
    for (int ts = 0; ts < T; ts += slab) {
        const int tiles = T - ts < slab ? T - ts : slab;
        if (!mma_plan(tiles, Ut, 2, active, &C, &G, &load)) return LBQ_ERR_SHAPE;
        const long long n0 = static_cast<long long>(ts) * kTileRows;
        const long long Ns = N - n0 < static_cast<long long>(tiles) * kTileRows ? N - n0
                                                                                 : static_cast<long long>(tiles) * kTileRows;
        MmaArgs a;
        std::memset(&a, 0, sizeof(a));
        a.blob = b;
        a.area = b + L.area_offset + (n0 / 4) * static_cast<long long>(L.row_block_bytes);
        a.x = static_cast<const __half*>(x);
        a.y = static_cast<uint8_t*>(y) + n0 * (y_f32 ? 4 : 2);
        a.err = err_word;
        a.ldx = ldx;
        a.ldy = ldy;
        a.N = Ns;
        a.K = K;
        a.N_hdr = N;
        a.rb_bytes = static_cast<long long>(L.row_block_bytes);
        a.n_rb = static_cast<int>((Ns + 3) / 4);
        a.T = tiles;
        a.U = U;
        a.Ud = Ud;
        a.OS = OS;
        a.Ut = Ut;
        a.n_out = n_out;
        a.OT = OT;
        a.recs = static_cast<int>(L.records);
        a.cols_last = cols_last;
        a.idx = n_out > 0 ? reinterpret_cast<const int32_t*>(b + L.idx_offset) : nullptr;
        a.C = C;
        a.G = G;
        a.M = M;
        a.Mr = (M + 7) / 8 * 8;
        a.y_f32 = y_f32 ? 1 : 0;
        a.lut_lo = lut_lo;
        a.lut_hi = lut_hi;
        // tensor map of X: (k, activation row), 64-k x Mr-row boxes in the MMA's swizzled layout
        Maps maps;
        std::memset(&maps, 0, sizeof(maps));
        const cuuint32_t one[2] = {1, 1};
        bool enc = true;
        {
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
            const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStageK), static_cast<cuuint32_t>(a.Mr)};
            enc = enc && encode(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box,
                                one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        // tensor maps of the outlier values, FP16 (column, row, [record,] row block):
        // 64-column x 256-row boxes in the MMA's swizzled layout; columns past the
        // last record's width and row blocks past the slab read as zero
        if (n_out > 0) {
            uint8_t* out0 = b + L.area_offset + (n0 / 4) * static_cast<long long>(L.row_block_bytes) +
                            L.records * L.record_bytes;
            const cuuint32_t one4[4] = {1, 1, 1, 1};
            if (OT > 1) {
                const cuuint64_t dims[4] = {static_cast<cuuint64_t>(lbq::kOutlierCols), 4,
                                            static_cast<cuuint64_t>(OT - 1), static_cast<cuuint64_t>(a.n_rb)};
                const cuuint64_t strides[3] = {static_cast<cuuint64_t>(lbq::kOutlierCols) * 2,
                                               static_cast<cuuint64_t>(L.outlier_record_bytes),
                                               static_cast<cuuint64_t>(L.row_block_bytes)};
                const cuuint32_t box[4] = {static_cast<cuuint32_t>(kStageK), 4, 1, static_cast<cuuint32_t>(kTileRb)};
                enc = enc && encode(&maps.out_full, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, out0, dims, strides, box, one4,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
            }
            const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols_last), 4, static_cast<cuuint64_t>(a.n_rb)};
            const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols_last) * 2,
                                           static_cast<cuuint64_t>(L.row_block_bytes)};
            const cuuint32_t box[3] = {static_cast<cuuint32_t>(kStageK), 4, static_cast<cuuint32_t>(kTileRb)};
            enc = enc && encode(&maps.out_last, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                                out0 + static_cast<long long>(OT - 1) * L.outlier_record_bytes, dims, strides, box,
                                one4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        if (!enc) return LBQ_ERR_CUDA;
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(static_cast<unsigned>(C * G));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr[2];
        int na = 0;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(C);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
        // later slabs follow a slab of this same call, which never writes the weights or x
        if ((flags & LBQ_FLAG_PDL) || ts > 0) {
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        cfg.attrs = attr;
        cfg.numAttrs = na;
        void* args[] = {&a, &maps};
        if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
            (void)cudaGetLastError();
            return LBQ_ERR_CUDA;
        }
    }
    return LBQ_OK;
}

}  // namespace lbq
