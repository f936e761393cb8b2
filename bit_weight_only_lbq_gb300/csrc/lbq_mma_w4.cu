// 4-bit small-M GEMM on the 5th-generation tensor cores (tcgen05) for
// M >= 16 activation rows, sm_103a.
//
// Method (SPECTRA article, section 4.2 "Batched Tensor Core W4A16 GEMM with
// In-Kernel Outlier Fusion"): at M >= 16 the product Y = X W_hat^T is a real
// dense contraction, so the packed 4-bit weights are dequantised in the kernel
// to FP16 tiles w_hat = s (q - z) and multiplied on the tensor cores with FP32
// accumulation; the weights still cross HBM once, in their packed form.
//
// GB300 design:
//  * a CTA owns a tile of 128 weight rows (32 row blocks of the blob) and a
//    range of its 1024-k record blocks, walked in 256-k stages;
//  * three tensor maps feed it through the Tensor Memory Accelerator: the
//    nibbles of one stage for the 32 row blocks x 4 rows (16 KB, 128-byte
//    swizzle, so the dequantising threads read shared memory without bank
//    conflicts), the scales and zero points of a record block (10 KB), and
//    the activations of the stage, written by the copy engine straight in the
//    128-byte-swizzled K-major layout the tensor core reads (rows past M and
//    columns past K arrive as zeros);
//  * warp roles: one warp copies the weights (nibbles and metadata, which no
//    earlier kernel writes, so it starts before the grid dependency resolves),
//    one copies the activations, two issue tcgen05.mma (alternate stages, each
//    into its own accumulator: a barrier wait holds the issuing thread until its
//    earlier MMAs are taken, and the other warp issues meanwhile), sixteen
//    dequantise - each thread owns one weight row (its tensor-memory lane) and
//    2 groups per stage: 1024 + q from the nibble masked into the FP16 magic
//    exponent, minus (1024 + z) exactly, times the FP16 scale (one rounding),
//    stored into tensor memory with tcgen05.st (k in natural order).  A stays in
//    tensor memory rather than shared memory: written and read there it would
//    cost 128 KB of shared-memory traffic per stage;
//  * every hand-off is an mbarrier: rings of 6-10 nibble stages, 2 metadata
//    blocks, 3-4 activation stages, and 3 A stages in tensor memory (freed by
//    tcgen05.commit when the tensor core has read them);
//  * tcgen05.mma: A from tensor memory (128 rows), B from shared memory
//    (N = 16..64 activation rows), K = 16, FP16 x FP16 -> FP32 in tensor
//    memory; the two accumulators are added in a fixed order at the end;
//  * when a tile's K is split over a cluster of CTAs, each CTA moves its FP32
//    partial from tensor memory to shared memory and the cluster's rank 0 adds
//    the partials in rank order through distributed shared memory
//    (deterministic, no global workspace);
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

constexpr int kWorkerWarps = 16;             // dequantising warps: 4 per tensor-memory lane quarter
constexpr int kWorkers = 32 * kWorkerWarps;
// tensor-core issue is split over two warps taking alternate stages, each into
// its own accumulator: a barrier wait holds its thread until the MMAs it issued
// before have been taken by the tensor core, and the other warp issues meanwhile
constexpr int kIssuers = 2;
constexpr int kThreads = kWorkers + 64 + 32 * kIssuers;   // + weight-copy, activation-copy and MMA warps
constexpr int kTileRows = 128;               // MMA M
constexpr int kTileRb = kTileRows / 4;       // row blocks per tile
constexpr int kRecBytes = 2368;              // 4-bit dense record
constexpr int kMetaBytes = 320;              // its scales (256) and zero points (64)
constexpr int kStageK = 256;                 // k per stage (8 groups)
constexpr int kStagesPerBlock = 1024 / kStageK;
constexpr int kGpw = 8 / (kWorkerWarps / 4);    // groups of a stage per dequantising warp
constexpr int kCodeStage = kTileRb * 4 * 128;   // 16 KB: 8 groups x 16 B for 128 rows
constexpr int kMetaBlock = kTileRb * kMetaBytes;  // 10 KB
constexpr int kNA = 3;                       // A stages in tensor memory
constexpr uint32_t kTmemCols = 512;          // accumulators in [0, 128), A stages from column 128
constexpr uint32_t kAcol = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct MmaArgs {
    const uint8_t* blob;
    void* y;
    unsigned* err;
    long long ldy;
    long long N, K;
    int recs;       // k-blocks
    int n_rb;
    int M;          // activation rows (<= NM)
    int S;          // k-splits per tile = cluster size
    int y_f32;
    // outlier columns, added in the epilogue: X (row-major, ldx), their channels,
    // and the outlier records (after the dense records of each row block)
    const __half* x;
    long long ldx;
    const int32_t* idx;
    int n_out;
    int OT;                 // outlier records per row block
    int cols_last;          // columns of the last one (a multiple of 8)
    long long rb_bytes;
    const uint8_t* out0;    // outlier records of row block 0
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
__device__ __forceinline__ uint32_t u4w(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Word j (0..3) of a group's 16 qweight bytes (byte k = q_k | q_{k+16} << 4) as
// 8 dequantised FP16 weights in natural order: lo[0] = (w_{4j}, w_{4j+1}),
// lo[1] = (w_{4j+2}, w_{4j+3}), hi[0] = (w_{4j+16}, w_{4j+17}), hi[1] = (w_{4j+18}, w_{4j+19}).
// 1024 + q is exact in FP16 (magic exponent), (1024 + q) - (1024 + z) = q - z
// exactly, (1024 + 16 q) / 16 - (64 + z) = q - z exactly, then one rounding by s.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zlo2, uint32_t zhi2, uint32_t s2, uint32_t (&lo)[2],
                                             uint32_t (&hi)[2]) {
    const uint32_t sixteenth2 = 0x2C002C00u;   // FP16 1/16 in both halves
    const uint32_t b01 = prmt(w, 0u, 0x4140u), b23 = prmt(w, 0u, 0x4342u);   // bytes 0,1 / 2,3 to the halves
    lo[0] = hmul2(hsub2((b01 & 0x000F000Fu) | 0x64006400u, zlo2), s2);
    lo[1] = hmul2(hsub2((b23 & 0x000F000Fu) | 0x64006400u, zlo2), s2);
    hi[0] = hmul2(hfma2((b01 & 0x00F000F0u) | 0x64006400u, sixteenth2, zhi2), s2);
    hi[1] = hmul2(hfma2((b23 & 0x00F000F0u) | 0x64006400u, sixteenth2, zhi2), s2);
}

template <int NM>
struct Geom {
    // stages in flight within 227 KB of shared memory: nibbles (16 KB each; the
    // deeper the better against DRAM latency) and activations (NM x 512 B each)
    static constexpr int kNC = NM == 16 ? 10 : NM <= 48 ? 8 : 6;
    static constexpr int kNB = NM <= 32 ? 4 : 3;
    static constexpr int kBBox = NM * 128;                         // one 64-k box of NM rows
    static constexpr int kBStage = 4 * kBBox;
    static constexpr int code = 0;                                 // kNC x 16 KB (1024-aligned)
    static constexpr int b = code + kNC * kCodeStage;              // kNB activation stages
    static constexpr int meta = b + kNB * kBStage;                 // 2 x 10 KB
    static constexpr int bars = meta + 2 * kMetaBlock;
    static constexpr int nbars = 2 * kNC + 2 * 2 + 2 * kNB + 2 * kNA + 1;
    static constexpr int total = bars + 8 * nbars + 32 + 1024;    // + flags, alignment
};

struct Maps {
    CUtensorMap codes, meta, x;
};

template <int NM>
__global__ void __launch_bounds__(kThreads, 1)
    lbq_w4_mma_kernel(const __grid_constant__ MmaArgs a, const __grid_constant__ Maps maps) {
    using G = Geom<NM>;
    constexpr int kNB = G::kNB;
    constexpr int kNC = G::kNC;
    constexpr uint32_t kIdesc = idesc_f16(kTileRows, NM);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::bars);
    // mbarriers: code full/empty [kNC], meta full/empty [2], b full/empty [kNB], a full/empty [kNA], last
    const uint32_t cfull = smem_u32(bars), cempty = cfull + 8 * kNC, mfull = cempty + 8 * kNC, mempty = mfull + 16,
                   bfull = mempty + 16, bempty = bfull + 8 * kNB, afull = bempty + 8 * kNB, aempty = afull + 8 * kNA,
                   last_bar = aempty + 8 * kNA;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + G::nbars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + G::nbars) + 1;
    // stages (nibbles, activations) and record blocks (metadata) whose copies were issued
    volatile int* issued = reinterpret_cast<volatile int*>(bars + G::nbars) + 2;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.S;
    const int rank = static_cast<int>(blockIdx.x) % S;         // rank in the cluster (cluster = S consecutive CTAs)
    const int tile = static_cast<int>(blockIdx.x) / S;
    const int kb0 = rank * a.recs / S, kb1 = (rank + 1) * a.recs / S;
    const int nkb = kb1 - kb0;
    const int nstages = nkb * kStagesPerBlock;
    const int rb0 = tile * kTileRb;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int i = 0; i < G::nbars; ++i) {
            const uint32_t bar = cfull + 8 * i;
            // arrivals: copies (1, with the byte count), the dequantising warps,
            // one tensor-core commit, or one commit per MMA warp (the last)
            const bool workers = (bar >= cempty && bar < mfull) || (bar >= mempty && bar < bfull) ||
                                 (bar >= afull && bar < aempty);
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
                         "r"(workers ? kWorkerWarps : bar == last_bar ? kIssuers : 1)
                         : "memory");
        }
        *abort_flag = 0;
        issued[0] = issued[1] = issued[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // bounded wait that gives up at once after any thread of the CTA gave up
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        // no sleep between polls: try_wait suspends the thread until the phase
        // completes or a short hardware limit passes, and a sleep would only add
        // wake-up latency to every hand-off
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
                return false;
            }
        }
        return true;
    };
    auto arrive = [&](uint32_t bar) {
        asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    };
    auto expect = [&](uint32_t bar, uint32_t bytes) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    };

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    auto commit = [&](uint32_t bar) {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    };
    if (warp == kWorkerWarps) {
        // ------------------------------------------------------------------ weight copies
        // the packed weights are not written by earlier kernels: no wait on them
        if (lane == 0) {
            int s = 0;
            for (; s < nstages; ++s) {
                const int kb = kb0 + s / kStagesPerBlock, sl = s % kStagesPerBlock, blk = s / kStagesPerBlock;
                if (sl == 0) {
                    const int m = blk & 1;
                    if (blk >= 2 && !wait(mempty + 8 * m, ((blk - 2) >> 1) & 1)) break;
                    expect(mfull + 8 * m, kMetaBlock);
                    asm volatile(
                        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem + G::meta + m * kMetaBlock)),
                        "l"(&maps.meta), "r"(0), "r"(kb), "r"(rb0), "r"(mfull + 8 * m)
                        : "memory");
                    issued[2] = blk + 1;
                }
                const int c = s % kNC;
                if (s >= kNC && !wait(cempty + 8 * c, ((s - kNC) / kNC) & 1)) break;
                expect(cfull + 8 * c, kCodeStage);
                asm volatile(
                    "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem + G::code + c * kCodeStage)),
                    "l"(&maps.codes), "r"(128 * sl), "r"(0), "r"(kb), "r"(rb0), "r"(cfull + 8 * c)
                    : "memory");
            }
            issued[0] = s;
        }
        __syncwarp();
    } else if (warp == kWorkerWarps + 1) {
        // ------------------------------------------------------------------ activation copies
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");   // x may be written by the previous kernel
            int s = 0;
            for (; s < nstages; ++s) {
                const int kb = kb0 + s / kStagesPerBlock, sl = s % kStagesPerBlock;
                const int bs = s % kNB;
                if (s >= kNB && !wait(bempty + 8 * bs, ((s - kNB) / kNB) & 1)) break;
                expect(bfull + 8 * bs, G::kBStage);
                const int k0 = kb * 1024 + sl * kStageK;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    asm volatile(
                        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + G::b + bs * G::kBStage + j * G::kBBox)),
                        "l"(&maps.x), "r"(k0 + 64 * j), "r"(0), "r"(bfull + 8 * bs)
                        : "memory");
            }
            issued[1] = s;
        }
        __syncwarp();
    } else if (warp >= kWorkerWarps + 2) {
        // ------------------------------------------------------------------ tensor-core issue
        // MMA warp iw takes stages iw, iw + kIssuers, ... into accumulator iw
        const int iw = warp - (kWorkerWarps + 2);
        if (lane == 0) {
            for (int s = iw; s < nstages; s += kIssuers) {
                const int as = s % kNA, bs = s % kNB;
                const bool ok = wait(afull + 8 * as, (s / kNA) & 1) && wait(bfull + 8 * bs, (s / kNB) & 1);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok && !*abort_flag) {
                    const uint32_t b0 = smem_u32(smem + G::b + bs * G::kBStage);
#pragma unroll
                    for (int ks = 0; ks < kStageK / 16; ++ks) {
                        const uint64_t db = smem_desc_sw128(b0 + (ks >> 2) * G::kBBox + (ks & 3) * 32);
                        const uint32_t acc = (s >= kIssuers || ks > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + NM * iw),
                            "r"(tmem + kAcol + 128u * as + 8u * ks), "l"(db), "r"(kIdesc), "r"(acc)
                            : "memory");
                    }
                }
                // always commit, so that every wait on these stages completes
                commit(aempty + 8 * as);
                commit(bempty + 8 * bs);
            }
            commit(last_bar);   // tracks every tensor-core operation this thread issued
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ dequantisation
        // thread owns tensor-memory lane m = 32 (warp % 4) + lane = weight row
        // 4 rb + r of the tile, rb = 8 (warp % 4) + 2 (lane / 8) + (lane / 4) % 2,
        // r = lane % 4: the 8 lanes of a quarter warp read 8 different 16-byte
        // bank groups of the swizzled nibble stage; groups kGpw (warp / 4) .. + kGpw - 1
        const int qd = warp & 3, gh = warp >> 2;
        const int rb = 8 * qd + 2 * (lane >> 3) + ((lane >> 2) & 1), r = lane & 3;
        const int row128 = rb * 4 + r;                              // 128-byte row of the nibble stage
        const uint32_t tlane = static_cast<uint32_t>(32 * qd) << 16;
        for (int s = 0; s < nstages; ++s) {
            const int sl = s % kStagesPerBlock, blk = s / kStagesPerBlock;
            const int c = s % kNC, as = s % kNA, m = blk & 1;
            // lane 0 polls for the warp; __syncwarp then orders the other lanes
            // after its acquire
            bool ok = true;
            if (lane == 0) {
                if (sl == 0) ok = wait(mfull + 8 * m, (blk >> 1) & 1) && ok;
                ok = wait(cfull + 8 * c, (s / kNC) & 1) && ok;
                if (s >= kNA) ok = wait(aempty + 8 * as, ((s - kNA) / kNA) & 1) && ok;
            }
            __syncwarp();
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (ok && !*abort_flag) {
                const uint8_t* cs = smem + G::code + c * kCodeStage + row128 * 128;
                const uint8_t* ms = smem + G::meta + m * kMetaBlock + rb * kMetaBytes;
                const int g0 = 8 * sl + kGpw * gh;                  // first of this thread's groups in the record
                static_assert(kGpw == 2, "scale and zero-point loads below are for two groups per warp");
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(ms + r * 64 + g0 * 2);   // 2 FP16 scales
                const uint32_t zw = ms[256 + r * 16 + g0 / 2];                                   // 2 zero points
#pragma unroll
                for (int t = 0; t < kGpw; ++t) {
                    const int g8 = kGpw * gh + t;                   // group of the stage
                    const uint4 q = *reinterpret_cast<const uint4*>(cs + ((g8 ^ (row128 & 7)) << 4));
                    const uint32_t z = (zw >> (4 * t)) & 15u;
                    const uint32_t sb = sc >> (16 * t) & 0xFFFFu;
                    const uint32_t zlo2 = (0x6400u | z) * 0x00010001u;           // 1024 + z
                    const uint32_t zhi2 = (0xD400u | (z << 4)) * 0x00010001u;    // -(64 + z)
                    const uint32_t s2 = sb * 0x00010001u;
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t lo[2], hi[2];
                        dequant_word(u4w(q, j), zlo2, zhi2, s2, lo, hi);
                        v[2 * j] = lo[0];
                        v[2 * j + 1] = lo[1];
                        v[8 + 2 * j] = hi[0];
                        v[9 + 2 * j] = hi[1];
                    }
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                        "%12, %13, %14, %15, %16};" ::"r"(tmem + tlane + kAcol + 128u * as + 16u * g8),
                        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                        : "memory");
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                arrive(cempty + 8 * c);                                 // this warp is done with the nibbles
                if (sl == kStagesPerBlock - 1) arrive(mempty + 8 * m);  // and with the block's metadata
                arrive(afull + 8 * as);
            }
        }
    }
    // the accumulator is complete once the last commit has arrived
    const bool got = nstages == 0 || mbar_wait(last_bar, 0, kWaitLimitNs);
    if (!got && tid == 0) atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
    __syncthreads();
    const bool bad = *abort_flag != 0 || !got;
    // after an abort, the last copies issued may still be in flight: wait for them
    // (a stage the copy warps never issued is not waited for)
    if (bad && tid == kWorkers) {
        const int ic = issued[0], ix = issued[1], im = issued[2];
        for (int s = ic > kNC ? ic - kNC : 0; s < ic; ++s)
            mbar_wait(cfull + 8 * (s % kNC), (s / kNC) & 1, kWaitLimitNs / 64);
        for (int s = ix > kNB ? ix - kNB : 0; s < ix; ++s)
            mbar_wait(bfull + 8 * (s % kNB), (s / kNB) & 1, kWaitLimitNs / 64);
        for (int blk = im > 2 ? im - 2 : 0; blk < im; ++blk)
            mbar_wait(mfull + 8 * (blk & 1), (blk >> 1) & 1, kWaitLimitNs / 64);
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // epilogue: warp w reads accumulator lanes 32 (w % 4) .. + 31 (its rows) and
    // columns 16 (w / 4) .. + 15 (activation rows), so up to 16 warps share it
    constexpr int kChunks = NM / 16;
    const int qd = warp & 3, cc = warp >> 2;
    const bool ep = warp < 4 * kChunks;
    const int m = 32 * qd + lane;
    const int erb = 8 * qd + 2 * (lane >> 3) + ((lane >> 2) & 1), er = lane & 3;
    const long long n = static_cast<long long>(rb0 + erb) * 4 + er;
    float d[16];
    if (ep) {
#pragma unroll
        for (int i = 0; i < 16; ++i) d[i] = 0.f;
#pragma unroll
        for (int acc = 0; acc < kIssuers; ++acc) {   // the accumulators, added in a fixed order
            uint32_t v[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                "%13, %14, %15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(tmem + (static_cast<uint32_t>(32 * qd) << 16) + NM * acc + 16 * cc));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 16; ++i) d[i] += (nstages > 0 && !bad) ? __uint_as_float(v[i]) : 0.f;
        }
    }
    auto write_y = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the previous kernel is done with y
        if (n < a.N && !bad) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int row = 16 * cc + i;
                if (row < a.M) {
                    if (a.y_f32)
                        reinterpret_cast<float*>(a.y)[row * a.ldy + n] = d[i];
                    else
                        reinterpret_cast<__half*>(a.y)[row * a.ldy + n] = __float2half_rn(d[i]);
                }
            }
        }
    };
    // exact FP16 outlier columns (SPECTRA section 4.2, in-kernel outlier fusion):
    // d[i] += sum_j X[16 cc + i][idx_j] Wout[n][j], in FP32, columns in order, by the
    // CTA's partial.  In chunks of 64 columns (chunks c0, c0 + cs, ...: with K
    // split over a cluster every rank adds its share of the chunks to its own
    // partial, which the rank-order reduction then sums): the chunk's X[:, idx] (NM rows,
    // zero past M) and the tile's outlier values of the chunk are staged in shared
    // memory by the whole CTA with every load in flight (one round trip to memory
    // per chunk), then each thread adds its row's 64 columns.
    auto add_outliers = [&](int c0, int cs) {
        if (a.n_out <= 0 || bad) return;
        // staging areas over the idle rings: the chunk's activations X[:, idx] as FP32
        // (activation ring), the outlier channels (once) and the tile's 128 rows x 64
        // FP16 outlier values of the chunk (nibble ring, past the split-K partials;
        // rows padded to 144 bytes: conflict-free 16-byte reads by row)
        float* xo = reinterpret_cast<float*>(smem + G::b);
        int* ids = reinterpret_cast<int*>(smem + G::code + 32768);
        uint8_t* wo = smem + G::code + 32768 + 4 * lbq::kMaxOutliers;
        constexpr int kWoRow = 144;
        static_assert(G::kNC * kCodeStage >= 32768 + 4 * lbq::kMaxOutliers + kTileRows * kWoRow,
                      "outlier staging fits the nibble ring");
        __syncthreads();   // every thread is past the partials' reads
        for (int j = tid; j < a.n_out; j += kThreads) {
            const int k = a.idx[j];
            const bool ok_k = k >= 0 && k < a.K;
            if (!ok_k) atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_OUTLIER_IDX));   // corrupted blob
            ids[j] = ok_k ? k : -1;
        }
        const int nrow = static_cast<int>(n - static_cast<long long>(rb0) * 4);   // this thread's tile row
        for (int j0 = 64 * c0; j0 < a.n_out; j0 += 64 * cs) {
            const int nj = min(64, a.n_out - j0);
            const int o = j0 / lbq::kOutlierCols, width = o + 1 < a.OT ? lbq::kOutlierCols : a.cols_last;
            __syncthreads();   // the channels are staged, the previous chunk has been read
            // the tile's outlier values of the chunk: 128 rows x 8 loads of 16 bytes, every
            // load in flight at once (zero padding past n_out within a record)
            for (int e = tid; e < kTileRows * 8; e += kThreads) {
                const int row = e >> 3, u = e & 7, rb = rb0 + (row >> 2);
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (rb < a.n_rb && 8 * u < nj)
                    v = *reinterpret_cast<const uint4*>(
                        a.out0 + static_cast<long long>(rb) * a.rb_bytes +
                        static_cast<long long>(o) * (lbq::kOutlierCols * lbq::kRowsPerBlock * 2) +
                        (static_cast<long long>(row & 3) * width + j0 % lbq::kOutlierCols + 8 * u) * 2);
                *reinterpret_cast<uint4*>(wo + row * kWoRow + 16 * u) = v;
            }
            for (int e = tid; e < NM * 64; e += kThreads) {
                const int row = e >> 6, j = j0 + (e & 63);
                float v = 0.f;
                if (row < a.M && j < a.n_out) {
                    const int k = ids[j];
                    if (k >= 0) v = __half2float(a.x[row * a.ldx + k]);
                }
                xo[e] = v;
            }
            __syncthreads();
            if (ep && n < a.N) {
                const float4* xo4 = reinterpret_cast<const float4*>(xo + 16 * cc * 64);
                const uint8_t* wr = wo + nrow * kWoRow;
#pragma unroll 1
                for (int u = 0; u < 8; ++u) {
                    if (8 * u >= nj) break;
                    const uint4 wv = *reinterpret_cast<const uint4*>(wr + 16 * u);   // 8 FP16 outlier values
                    const float2 w0 = __half22float2(*reinterpret_cast<const __half2*>(&wv.x));
                    const float2 w1 = __half22float2(*reinterpret_cast<const __half2*>(&wv.y));
                    const float2 w2 = __half22float2(*reinterpret_cast<const __half2*>(&wv.z));
                    const float2 w3 = __half22float2(*reinterpret_cast<const __half2*>(&wv.w));
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 xa = xo4[i * 16 + 2 * u], xb = xo4[i * 16 + 2 * u + 1];
                        float t = d[i];
                        t = fmaf(w0.x, xa.x, t);
                        t = fmaf(w0.y, xa.y, t);
                        t = fmaf(w1.x, xa.z, t);
                        t = fmaf(w1.y, xa.w, t);
                        t = fmaf(w2.x, xb.x, t);
                        t = fmaf(w2.y, xb.y, t);
                        t = fmaf(w3.x, xb.z, t);
                        t = fmaf(w3.y, xb.w, t);
                        d[i] = t;
                    }
                }
            }
        }
    };
    if (S == 1) {
        add_outliers(0, 1);
        if (ep) write_y();
    } else {
        add_outliers(rank, S);
        // split K: partials through distributed shared memory, added in rank order by rank 0
        float* part = reinterpret_cast<float*>(smem + G::code);   // NM x 128 FP32 over the (idle) nibble ring
        if (ep)
#pragma unroll
            for (int i = 0; i < 16; ++i) part[(16 * cc + i) * kTileRows + m] = d[i];
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (rank == 0) {
            if (ep)
                for (int p = 1; p < S; ++p) {
                    uint32_t remote;
                    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(part)), "r"(p));
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float v;
                        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                                     : "=f"(v)
                                     : "r"(remote + 4u * ((16 * cc + i) * kTileRows + m)));
                        d[i] += v;
                    }
                }
            if (ep) write_y();
        }
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    if (blockIdx.x == 0 && tid == 0) {
        const uint4* h = reinterpret_cast<const uint4*>(a.blob);
        const uint4 h0 = h[0], h1 = h[1], h2 = h[2];
        const long long n_hdr = (static_cast<long long>(h1.y) << 32) | h1.x;
        const long long k_hdr = (static_cast<long long>(h1.w) << 32) | h1.z;
        if (h0.x != 0x5751424Cu || h0.y != 0x32334734u || h0.z != LBQ_FORMAT_VERSION_NUM || n_hdr != a.N ||
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

template <int NM>
const void* kernel_fn() {
    return reinterpret_cast<const void*>(&lbq_w4_mma_kernel<NM>);
}

template <int NM>
int smem_bytes() {
    return Geom<NM>::total;
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

}  // namespace

namespace lbq {

int mma_padded_rows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : 64; }

// Launch the tensor-core 4-bit GEMM for one problem (16 <= M <= 64, no outlier
// columns).  Tiles of 128 rows; K split over a cluster of S CTAs so that tiles
// x S fills the SMs.  Returns LBQ_ERR_SHAPE when it does not fit.
lbq_status launch_w4_mma(const void* packed, int64_t N, int64_t K, int32_t n_out, int M, const void* x, int64_t ldx,
                         void* y, int64_t ldy, bool y_f32, unsigned* err_word, int sms, int max_smem, void* stream,
                         uint32_t flags) {
    if (M < 16 || M > 64) return LBQ_ERR_SHAPE;
    lbq_layout L;
    lbq_status st = lbq_blob_layout(LBQ_KIND_W4, N, K, n_out, &L);
    if (st != LBQ_OK) return st;
    const int NM = mma_padded_rows(M);
    const int smem = NM == 16 ? smem_bytes<16>() : NM == 32 ? smem_bytes<32>() : NM == 48 ? smem_bytes<48>()
                                                                                         : smem_bytes<64>();
    if (smem > max_smem) return LBQ_ERR_SHAPE;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
    if (!encode) return LBQ_ERR_CUDA;
    MmaArgs a;
    std::memset(&a, 0, sizeof(a));
    uint8_t* b = static_cast<uint8_t*>(const_cast<void*>(packed));
    a.blob = b;
    a.y = y;
    a.err = err_word;
    a.ldy = ldy;
    a.N = N;
    a.K = K;
    a.recs = static_cast<int>(L.records);
    a.n_rb = static_cast<int>((N + 3) / 4);
    a.M = M;
    a.y_f32 = y_f32 ? 1 : 0;
    a.x = static_cast<const __half*>(x);
    a.ldx = ldx;
    a.n_out = n_out;
    if (n_out > 0) {
        a.idx = reinterpret_cast<const int32_t*>(b + L.idx_offset);
        a.OT = static_cast<int>(L.outlier_records);
        a.cols_last = (n_out + lbq::kOutlierColAlign - 1) / lbq::kOutlierColAlign * lbq::kOutlierColAlign -
                      (a.OT - 1) * lbq::kOutlierCols;
        a.rb_bytes = static_cast<long long>(L.row_block_bytes);
        a.out0 = b + L.area_offset + L.records * L.record_bytes;
    }
    // tensor maps: nibbles (byte of a row's codes, row, record block, row block),
    // metadata (u16 of a record's scales + zeros, record block, row block),
    // activations (k, activation row)
    static thread_local Maps maps;
    std::memset(&maps, 0, sizeof(maps));
    const cuuint32_t one[4] = {1, 1, 1, 1};
    {
        const cuuint64_t dims[4] = {512, 4, static_cast<cuuint64_t>(a.recs), static_cast<cuuint64_t>(a.n_rb)};
        const cuuint64_t strides[3] = {512, static_cast<cuuint64_t>(kRecBytes), L.row_block_bytes};
        const cuuint32_t box[4] = {128, 4, 1, static_cast<cuuint32_t>(kTileRb)};
        if (encode(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, b + L.area_offset, dims, strides, box, one,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LBQ_ERR_CUDA;
    }
    {
        const cuuint64_t dims[3] = {kMetaBytes / 2, static_cast<cuuint64_t>(a.recs), static_cast<cuuint64_t>(a.n_rb)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRecBytes), L.row_block_bytes};
        const cuuint32_t box[3] = {kMetaBytes / 2, 1, static_cast<cuuint32_t>(kTileRb)};
        if (encode(&maps.meta, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, b + L.area_offset + 2048, dims, strides, box, one,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LBQ_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(NM)};
        if (encode(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, one,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return LBQ_ERR_CUDA;
    }
    const int tiles = (a.n_rb + kTileRb - 1) / kTileRb;
    int S = sms / tiles;
    if (S < 1) S = 1;
    if (S > 8) S = 8;
    if (S > a.recs) S = a.recs;
    a.S = S;
    const void* fn = NM == 16 ? kernel_fn<16>() : NM == 32 ? kernel_fn<32>() : NM == 48 ? kernel_fn<48>()
                                                                                      : kernel_fn<64>();
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return LBQ_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(S);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (flags & LBQ_FLAG_PDL) {
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
    return LBQ_OK;
}

}  // namespace lbq
