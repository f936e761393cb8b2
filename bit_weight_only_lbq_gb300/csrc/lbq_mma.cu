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
//    range of its 1024-k blocks; the 32 records of a k-block arrive by 32 bulk
//    copies into slots 2384 bytes apart (16 bytes of padding, so 8 consecutive
//    slots start in 8 different shared-memory bank groups), double buffered;
//  * per 256-k stage every thread dequantises 4 groups of one weight row:
//    nibbles masked with the FP16 magic 1024 (exact 1024 + q), minus (1024 + z),
//    times the FP16 scale (one rounding), stored straight into its row (lane)
//    of tensor memory with tcgen05.st - the A operand never touches shared
//    memory; the activations of the stage are staged in shared memory in the
//    no-swizzle K-major core-matrix layout (8 rows x 16 bytes per core matrix)
//    with the same permutation of k inside each group;
//  * one thread issues tcgen05.mma (A from tensor memory, M = 128 rows,
//    N = 16..64 activation rows, K = 16, FP16 x FP16 -> FP32 in tensor memory)
//    and tcgen05.commit to an mbarrier that frees the stage (double buffered);
//  * when a tile's K is split over a cluster of CTAs, each CTA moves its FP32
//    partial from tensor memory to shared memory and the cluster's rank 0 adds
//    the partials in rank order through distributed shared memory
//    (deterministic, no global workspace);
//  * every wait is bounded (2 s of %globaltimer); a timeout records
//    LBQ_ERR_TIMEOUT, the CTA drains its copies and tensor-core work, frees its
//    tensor memory and returns.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kTileRows = 128;            // MMA M
constexpr int kTileRb = kTileRows / 4;    // row blocks per tile
constexpr int kRecBytes = 2368;           // 4-bit dense record
constexpr int kSlot = 2384;               // shared-memory stride of a record slot
constexpr int kStageK = 256;              // k per A/B stage (8 groups)
constexpr int kStagesPerBlock = 1024 / kStageK;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct MmaArgs {
    const uint8_t* blob;
    const uint8_t* area;
    const __half* x;
    void* y;
    unsigned* err;
    long long ldx, ldy;
    long long N, K;
    long long rb_bytes;
    int recs;       // k-blocks
    int n_rb;
    int M;          // activation rows (<= NM)
    int S;          // k-splits per tile = cluster size
    int y_f32;
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
    for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
        __nanosleep(128);
    }
    return true;
}

// UMMA shared-memory descriptor, K-major without swizzle: core matrices of
// 8 rows x 16 bytes; `lbo` bytes between core matrices along K, `sbo` bytes
// between core matrices along M/N; version 1 (tcgen05).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;                      // descriptor version for tcgen05
    return d;                             // base offset 0, layout type 0 (no swizzle)
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

// Word j (0..3) of a group's 16 qweight bytes (byte k = q_k | q_{k+16} << 4)
// as 8 dequantised FP16 weights, in the order
//   (w_{4j}, w_{4j+2}), (w_{4j+1}, w_{4j+3}), (w_{4j+16}, w_{4j+18}), (w_{4j+17}, w_{4j+19}):
// 1024 + q is exact in FP16 (magic exponent), (1024 + q) - (1024 + z) = q - z exactly,
// (1024 + 16 q) / 16 - (64 + z) = q - z exactly, then one rounding by s.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t zlo2, uint32_t zhi2, uint32_t s2) {
    const uint32_t w8 = w >> 8;
    const uint32_t sixteenth2 = 0x2C002C00u;   // FP16 1/16 in both halves
    uint4 o;
    o.x = hmul2(hsub2((w & 0x000F000Fu) | 0x64006400u, zlo2), s2);
    o.y = hmul2(hsub2((w8 & 0x000F000Fu) | 0x64006400u, zlo2), s2);
    o.z = hmul2(hfma2((w & 0x00F000F0u) | 0x64006400u, sixteenth2, zhi2), s2);
    o.w = hmul2(hfma2((w8 & 0x00F000F0u) | 0x64006400u, sixteenth2, zhi2), s2);
    return o;
}

// The activations of one group in the same order, chunk j of 16 natural pairs
// n_i = (x_{2i}, x_{2i+1}).
__device__ __forceinline__ uint4 x_chunk(const uint32_t (&n)[16], int j) {
    uint4 c;
    c.x = prmt(n[2 * j], n[2 * j + 1], 0x5410u);
    c.y = prmt(n[2 * j], n[2 * j + 1], 0x7632u);
    c.z = prmt(n[8 + 2 * j], n[9 + 2 * j], 0x5410u);
    c.w = prmt(n[8 + 2 * j], n[9 + 2 * j], 0x7632u);
    return c;
}

struct Smem {
    static constexpr int kRecBuf = kTileRb * kSlot;            // one k-block of records
    static constexpr int rec = 0;
    static constexpr int b = 2 * kRecBuf;                      // 2 activation (B) stages
    static __host__ __device__ constexpr int bstage(int nm) { return nm * kStageK * 2; }
    static __host__ __device__ constexpr int bars(int nm) { return b + 2 * bstage(nm); }
    static __host__ __device__ constexpr int total(int nm) { return bars(nm) + 128 + 1024; }   // + alignment slack
};

// Tensor memory: columns [0, 64) the FP32 accumulator (128 lanes x N), then two
// A stages of 128 columns (128 rows x 256 FP16 k, two k per 32-bit column).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 128;

template <int NM>
__global__ void __launch_bounds__(kThreads + 32, 1) lbq_w4_mma_kernel(const __grid_constant__ MmaArgs a) {
    constexpr int kBStage = Smem::bstage(NM);
    constexpr int kSbo = (kStageK / 8) * 128;                   // bytes between 8-row groups of a B stage
    constexpr uint32_t kIdesc = idesc_f16(kTileRows, NM);
    constexpr int kWorkerWarps = kThreads / 32;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* recbuf = smem + Smem::rec;
    uint8_t* bbuf = smem + Smem::b;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars(NM));
    // mbarriers: full[2] records landed, ready[2] stage written, mdone[2] stage
    // consumed by the tensor core, rfree[2] record buffer read, last
    const uint32_t full0 = smem_u32(bars + 0), ready0 = smem_u32(bars + 2), mdone0 = smem_u32(bars + 4),
                   rfree0 = smem_u32(bars + 6), last_bar = smem_u32(bars + 8);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 10);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool mma_warp = warp == kWorkerWarps;                 // warp 8: copies and tensor-core issue
    const int S = a.S;
    const int rank = static_cast<int>(blockIdx.x) % S;         // rank in the cluster (cluster = S consecutive CTAs)
    const int tile = static_cast<int>(blockIdx.x) / S;
    const int kb0 = rank * a.recs / S, kb1 = (rank + 1) * a.recs / S;
    const int nkb = kb1 - kb0;
    const int rb0 = tile * kTileRb;
    const int nvalid = min(kTileRb, a.n_rb - rb0);
    const int nstages = nkb * kStagesPerBlock;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        const uint32_t counts[9] = {1, 1, kWorkerWarps, kWorkerWarps, 1, 1, kWorkerWarps, kWorkerWarps, 1};
        for (int i = 0; i < 9; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bars + i)), "r"(counts[i]) : "memory");
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // bounded wait that gives up at once after any thread of the CTA gave up
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
                return false;
            }
            __nanosleep(128);
        }
        return true;
    };
    auto arrive = [&](uint32_t bar) {
        asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    };

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (mma_warp) {
        // ---------------------------------------------------------------- copies + tensor-core issue
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        auto issue_block = [&](int kb, int bi) {
            const uint32_t bar = full0 + 8 * bi;
            if (lane == 0)
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                             "r"(static_cast<uint32_t>(nvalid * kRecBytes))
                             : "memory");
            __syncwarp();
            if (lane < nvalid) {
                const uint8_t* src = a.area + static_cast<long long>(rb0 + lane) * a.rb_bytes +
                                     static_cast<long long>(kb) * kRecBytes;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                    " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(recbuf + bi * Smem::kRecBuf + lane * kSlot)),
                    "l"(src), "r"(static_cast<uint32_t>(kRecBytes)), "r"(bar), "l"(policy)
                    : "memory");
            }
        };
        int issued = 0;
        for (; issued < 2 && issued < nkb; ++issued) issue_block(kb0 + issued, issued);
        for (int gs = 0; gs < nstages; ++gs) {
            const int ab = gs & 1;
            const bool ok = wait(ready0 + 8 * ab, (gs >> 1) & 1);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (lane == 0) {
                if (ok && !*abort_flag) {
                    const uint32_t b0 = smem_u32(bbuf + ab * kBStage);
#pragma unroll
                    for (int ks = 0; ks < kStageK / 16; ++ks) {
                        const uint64_t db = smem_desc(b0 + ks * 256, 128, kSbo);
                        const uint32_t acc = (gs > 0 || ks > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
                            "r"(tmem + kAcol + 128u * ab + 8u * ks), "l"(db), "r"(kIdesc), "r"(acc)
                            : "memory");
                    }
                }
                // always commit, so the workers' waits on this stage complete
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 mdone0 + 8 * ab)
                             : "memory");
            }
            __syncwarp();
            // after the last stage of k-block b: refill its record buffer with k-block b + 2
            if ((gs + 1) % kStagesPerBlock == 0) {
                const int b = gs / kStagesPerBlock;
                const bool freed = wait(rfree0 + 8 * (b & 1), (b >> 1) & 1);
                if (freed && !*abort_flag && issued < nkb) {
                    issue_block(kb0 + issued, issued & 1);
                    ++issued;
                }
            }
        }
        if (lane == 0)   // tracks every tensor-core operation issued before it
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(last_bar)
                         : "memory");
        __syncwarp();
        // drain: copies issued but never waited for by the workers (only after an abort)
        if (*abort_flag)
            for (int b = 0; b < issued; ++b) mbar_wait(full0 + 8 * (b & 1), (b >> 1) & 1, kWaitLimitNs / 8);
    } else {
        // ---------------------------------------------------------------- workers: activations + dequantisation
        asm volatile("griddepcontrol.wait;" ::: "memory");   // x may be written by the previous kernel
        // activation staging: NM rows x 8 groups per stage; thread takes tasks
        // tid, tid + 256, ... (row xa = task % NM, group task / NM)
        constexpr int kXTasks = NM * (kStageK / 32);
        constexpr int kXPer = (kXTasks + kThreads - 1) / kThreads;
        // two stages of activations in flight in registers (the stage loop below is
        // unrolled, so the buffer index s & 1 is a compile-time constant)
        uint4 xr[2][kXPer][4];
        auto load_x = [&](uint4 (&dst)[kXPer][4], int g) {       // stage g of this CTA
            const int kb = kb0 + g / kStagesPerBlock, s = g % kStagesPerBlock;
#pragma unroll
            for (int u = 0; u < kXPer; ++u) {
                const int task = tid + u * kThreads;
                const int xg = task / NM, xa = task - xg * NM;
                const long long k = static_cast<long long>(kb) * 1024 + s * kStageK + xg * 32;
#pragma unroll
                for (int c = 0; c < 4; ++c) dst[u][c] = make_uint4(0u, 0u, 0u, 0u);
                if (g < nstages && task < kXTasks && xa < a.M && k < a.K) {
                    const uint4* p = reinterpret_cast<const uint4*>(a.x + xa * a.ldx + k);
#pragma unroll
                    for (int c = 0; c < 4; ++c) dst[u][c] = p[c];
                }
            }
        };
        load_x(xr[0], 0);
        load_x(xr[1], 1);
        // dequant tasks: thread owns MMA row m = 32 (warp % 4) + lane = weight row
        // 4 (8 (warp % 4) + lane % 8) + lane / 8 of the tile (tensor-memory lane m)
        // and groups 4 (warp / 4) .. + 3 of each stage
        const int qd = warp & 3, gh = warp >> 2;
        const int slot = 8 * qd + (lane & 7), r = lane >> 3;
        const uint32_t tlane = static_cast<uint32_t>(32 * qd) << 16;
        int gs = 0;
        for (int b = 0; b < nkb; ++b) {
            const int bi = b & 1;
            const bool have = wait(full0 + 8 * bi, (b >> 1) & 1);
            const uint8_t* rec = recbuf + bi * Smem::kRecBuf + slot * kSlot;
#pragma unroll
            for (int s = 0; s < kStagesPerBlock; ++s, ++gs) {
                const int ab = gs & 1;
                bool ok = have;
                if (gs >= 2) ok = wait(mdone0 + 8 * ab, ((gs - 2) >> 1) & 1) && ok;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (ok && !*abort_flag) {
                    uint8_t* B = bbuf + ab * kBStage;
                    // activations of this stage (prefetched), then prefetch the next stage's
#pragma unroll
                    for (int u = 0; u < kXPer; ++u) {
                        const int task = tid + u * kThreads;
                        if (task < kXTasks) {
                            const int xg = task / NM, xa = task - xg * NM;
                            uint32_t n[16];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                n[4 * c + 0] = xr[s & 1][u][c].x;
                                n[4 * c + 1] = xr[s & 1][u][c].y;
                                n[4 * c + 2] = xr[s & 1][u][c].z;
                                n[4 * c + 3] = xr[s & 1][u][c].w;
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                *reinterpret_cast<uint4*>(B + (xa >> 3) * kSbo + (4 * xg + j) * 128 + (xa & 7) * 16) =
                                    x_chunk(n, j);
                        }
                    }
                    load_x(xr[s & 1], gs + 2);
                    // weights: 4 groups of row m into tensor memory, 16 columns each
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int gi = 4 * gh + t;                       // group of the stage
                        const int g = (kStageK / 32) * s + gi;           // group of the record
                        const uint4 q = *reinterpret_cast<const uint4*>(rec + (r * 32 + g) * 16);
                        const uint32_t sb = *reinterpret_cast<const unsigned short*>(rec + 2048 + (r * 32 + g) * 2);
                        const uint32_t zb = rec[2304 + r * 16 + (g >> 1)];
                        const uint32_t z = (g & 1) ? (zb >> 4) : (zb & 15u);
                        const uint32_t zlo2 = (0x6400u | z) * 0x00010001u;           // 1024 + z
                        const uint32_t zhi2 = (0xD400u | (z << 4)) * 0x00010001u;    // -(64 + z)
                        const uint32_t s2 = sb * 0x00010001u;
                        uint4 o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) o[j] = dequant_word(u4w(q, j), zlo2, zhi2, s2);
                        asm volatile(
                            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
                            "%11, %12, %13, %14, %15, %16};" ::"r"(tmem + tlane + kAcol + 128u * ab + 16u * gi),
                            "r"(o[0].x), "r"(o[0].y), "r"(o[0].z), "r"(o[0].w), "r"(o[1].x), "r"(o[1].y), "r"(o[1].z),
                            "r"(o[1].w), "r"(o[2].x), "r"(o[2].y), "r"(o[2].z), "r"(o[2].w), "r"(o[3].x), "r"(o[3].y),
                            "r"(o[3].z), "r"(o[3].w)
                            : "memory");
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if (s + 1 == kStagesPerBlock) arrive(rfree0 + 8 * bi);  // this warp is done with the records
                    arrive(ready0 + 8 * ab);
                }
            }
        }
    }
    // the accumulator is complete once the last commit has arrived
    const bool got = nstages == 0 || mbar_wait(last_bar, 0, kWaitLimitNs);
    if (!got && tid == 0) atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_TIMEOUT));
    __syncthreads();
    const bool bad = *abort_flag != 0 || !got;
    const int gs = nstages;
    const int qd = warp & 3;
    const int m = 32 * qd + lane;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // epilogue: warps 0-3 read rows 32 w .. 32 w + 31 of the accumulator
    float d[NM];
    if (warp < 4) {
#pragma unroll
        for (int c = 0; c < NM / 16; ++c) {
            uint32_t v[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                "%14, %15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 16 * c));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 16; ++i) d[16 * c + i] = (gs > 0 && !bad) ? __uint_as_float(v[i]) : 0.f;
        }
    }
    const long long n = static_cast<long long>(rb0 + 8 * qd + (lane & 7)) * 4 + (lane >> 3);
    auto write_y = [&](const float (&dv)[NM]) {
        if (n < a.N && !bad) {
#pragma unroll
            for (int i = 0; i < NM; ++i) {
                if (i < a.M) {
                    if (a.y_f32)
                        reinterpret_cast<float*>(a.y)[i * a.ldy + n] = dv[i];
                    else
                        reinterpret_cast<__half*>(a.y)[i * a.ldy + n] = __float2half_rn(dv[i]);
                }
            }
        }
    };
    if (S == 1) {
        if (warp < 4) write_y(d);
    } else {
        // split K: partials through distributed shared memory, added in rank order by rank 0
        float* part = reinterpret_cast<float*>(recbuf);           // 128 x NM FP32, record buffers are free
        if (warp < 4)
#pragma unroll
            for (int i = 0; i < NM; ++i) part[i * kTileRows + m] = d[i];
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (rank == 0 && warp < 4) {
            for (int p = 1; p < S; ++p) {
                uint32_t remote;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(part)), "r"(p));
#pragma unroll
                for (int i = 0; i < NM; ++i) {
                    float v;
                    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote + 4u * (i * kTileRows + m)));
                    d[i] += v;
                }
            }
            write_y(d);
        }
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    if (blockIdx.x == 0 && tid == 0) {
        const uint4* h = reinterpret_cast<const uint4*>(a.blob);
        const uint4 h0 = h[0], h1 = h[1], h2 = h[2];
        const long long n_hdr = (static_cast<long long>(h1.y) << 32) | h1.x;
        const long long k_hdr = (static_cast<long long>(h1.w) << 32) | h1.z;
        if (h0.x != 0x5751424Cu || h0.y != 0x32334734u || h0.z != LBQ_FORMAT_VERSION_NUM || n_hdr != a.N ||
            k_hdr != a.K || h2.x != 0u)
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

}  // namespace

namespace lbq {

int mma_padded_rows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : 64; }

// Launch the tensor-core 4-bit GEMM for one problem (16 <= M <= 64, no outlier
// columns).  Tiles of 128 rows; K split over a cluster of S CTAs so that tiles
// x S fills the SMs.  Returns LBQ_ERR_SHAPE when it does not fit.
lbq_status launch_w4_mma(const void* packed, int64_t N, int64_t K, int M, const void* x, int64_t ldx, void* y,
                         int64_t ldy, bool y_f32, unsigned* err_word, int sms, int max_smem, void* stream,
                         uint32_t flags) {
    if (M < 16 || M > 64) return LBQ_ERR_SHAPE;
    lbq_layout L;
    lbq_status st = lbq_blob_layout(LBQ_KIND_W4, N, K, 0, &L);
    if (st != LBQ_OK) return st;
    const int NM = mma_padded_rows(M);
    const int smem = NM == 16 ? Smem::total(16) : NM == 32 ? Smem::total(32) : NM == 48 ? Smem::total(48) : Smem::total(64);
    if (smem > max_smem) return LBQ_ERR_SHAPE;
    MmaArgs a;
    std::memset(&a, 0, sizeof(a));
    const uint8_t* b = static_cast<const uint8_t*>(packed);
    a.blob = b;
    a.area = b + L.area_offset;
    a.x = static_cast<const __half*>(x);
    a.y = y;
    a.err = err_word;
    a.ldx = ldx;
    a.ldy = ldy;
    a.N = N;
    a.K = K;
    a.rb_bytes = static_cast<long long>(L.row_block_bytes);
    a.recs = static_cast<int>(L.records);
    a.n_rb = static_cast<int>((N + 3) / 4);
    a.M = M;
    a.y_f32 = y_f32 ? 1 : 0;
    const int tiles = (a.n_rb + kTileRb - 1) / kTileRb;
    int S = sms / tiles;
    if (S < 1) S = 1;
    if (S > 8) S = 8;
    if (S > a.recs) S = a.recs;
    a.S = S;
    const void* fn = NM == 16 ? kernel_fn<16>() : NM == 32 ? kernel_fn<32>() : NM == 48 ? kernel_fn<48>() : kernel_fn<64>();
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return LBQ_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * S));
    cfg.blockDim = dim3(kThreads + 32);
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
    void* args[] = {&a};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    return LBQ_OK;
}

}  // namespace lbq
