// Fused Group-32 low-bit decode GEMV kernels for sm_103a (GB300), and their
// C-ABI launchers.
//
// Method (SPECTRA article, section 4.1 "In-Register Fused W4A16 GEMV with
// Outlier Channel Accumulation"; otf-llm 4.0.0, section 5 and the
// "Architecture & Key Innovations" diagram): every packed weight is read
// once from HBM, unpacked in registers, combined with its group's
// scale/zero (4-bit) or codebook/S/Z (2-bit), multiplied with the FP16
// activation and accumulated in FP32; the exact FP16 outlier columns are
// accumulated into the same registers.
//
// GB300 design (the pages' kernels are Triton code for Ampere laptops):
//  * one launch serves a group of independent problems (a layer's linears, or
//    a list of them); their row blocks (4 output rows, all of K) form one
//    sequence that a persistent grid of <= one CTA per SM cuts into
//    contiguous, byte-balanced ranges;
//  * the blob stores each (4-row block x 32-group block) as one contiguous
//    record (packed codes, then scales/S, then zeros/Z); a CTA's items
//    (records and outlier records) are cut into contiguous per-warp ranges
//    (split-K inside the CTA when it owns few row blocks);
//  * each warp owns a private ring of shared-memory stages that its lane 0
//    refills with one bulk copy per item (cp.async.bulk, the Tensor Memory
//    Accelerator's 1-D mode) completing on an mbarrier; the warp moves an item
//    into registers and hands the stage back before computing on it, so every
//    stage but the one just read stays in flight;
//  * 4-bit: a nibble masked in place is an exact FP16 subnormal (q * 2^-24);
//    a mixed-precision FMA (FP16 inputs, exact FP32 product) accumulates
//    q * x in FP32, and the zero point enters once per group as z * sum(x);
//  * 2-bit: a byte-permute (PRMT) table lookup turns 2-bit codes into FP16
//    codebook values; S multiplies the codebook dot product, Z the group's
//    activation sum;
//  * outlier columns are streamed as extra 4 x 256 FP16 items of the same row
//    block and accumulated before the cross-lane reduction;
//  * partial rows of row blocks shared by several warps are combined in warp
//    order, so results do not depend on timing;
//  * every wait is bounded (2 s of %globaltimer); a timeout records
//    LBQ_ERR_TIMEOUT in a device error word and the warp drains its copies.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

__device__ unsigned int g_lbq_error_word;

constexpr int kTR = 4;                                 // output rows per row block
constexpr int kOutCols = 256;                          // outlier columns per outlier record
constexpr int kOutRecBytes = kTR * kOutCols * 2;       // 2048
constexpr int kMaxStagesPerWarp = 8;
// Deeper per-warp rings than this only delay every warp's first item (the copies
// of all warps queue together) without raising the streaming rate: measured on
// GB300, one-record stages, 16 warps.
constexpr int kStagesM1 = 2, kStagesMB = 4;
constexpr int kMaxGroup = LBQ_MAX_GROUP;               // problems per launch
constexpr int kMaxGrid = 192;                          // CTAs per launch (>= SMs of a GB300)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kRefineBatchMax = 512;                   // refinement columns staged at once per CTA

enum Kind { kW4 = 0, kW2 = 1 };

// Dense record geometry (one row block x 32 groups, the blob's unit); lane g
// of a warp owns group g of each of the record's 4 rows.
template <int KIND>
struct Rec {
    static constexpr int kPacked = KIND == kW4 ? 16 : 8;               // packed bytes per (row, group)
    static constexpr int kOff1 = kTR * 32 * kPacked;                   // scales / S
    static constexpr int kOff2 = kOff1 + kTR * 32 * 2;                 // zeros / Z
    static constexpr int kBytes = kOff2 + (KIND == kW4 ? kTR * 16 : kTR * 32 * 2);   // 2368 / 1536
    // a stage holds one item: RPI consecutive records of a row block, or one outlier record
    template <int RPI>
    static __host__ __device__ constexpr int stage() { return RPI * kBytes > kOutRecBytes ? RPI * kBytes : kOutRecBytes; }
    static constexpr uint32_t kMagicLo = 0x5751424Cu;                            // "LBQW"
    static constexpr uint32_t kMagicHi = KIND == kW4 ? 0x32334734u : 0x32334332u;  // "4G32" / "2C32"
};

// One problem of a launch (launch parameter space, read through the constant cache).
struct ProbArg {
    const uint8_t* blob;
    const uint8_t* area;   // first row block
    const int32_t* idx;
    const __half* x;       // activation rows, leading dimension ldx (elements)
    void* y;               // output rows, leading dimension ldy (elements)
    long long ldx, ldy;
    long long N, K;
    long long rb_bytes;    // bytes per row block
    int recs;              // dense records per row block
    int OT;                // outlier records per row block
    int out_last;          // bytes of the last one (4 rows x its columns, rounded up to 8, x 2 B)
    int n_out;
    int ub;                // index of its first row block in the launch's sequence
    // selective refinement (M = 1): blob of (N, K), its n_sel chosen channels, column bytes
    const uint8_t* rblob;  // or nullptr
    const int32_t* ridx;
    int nsel;
    long long rcb;
};

struct GroupArgs {
    int count;             // problems
    int nunits;            // row blocks of all problems
    int mrows;             // activation rows in this launch (<= MB of the kernel)
    int y_f32;
    int SPW;               // stages per warp
    int rb_cap;            // most row blocks any CTA owns
    int rearly;            // refinement pieces staged before the main loop (after the CTA's staging)
    uint32_t lut_lo, lut_hi;   // 2-bit codebook: low / high bytes of the FP16 centroids
    int cta_ub[kMaxGrid + 1];  // CTA c owns row blocks [cta_ub[c], cta_ub[c + 1])
    ProbArg p[kMaxGroup];
};

// ----------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false after the limit.
__device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
        __nanosleep(256);
    }
    return true;
}

// Lane 0 of the warp (the others skip it): arm the stage's mbarrier with the
// byte count and start the copy.  All lanes execute this code path, so the
// bookkeeping around it stays warp-uniform.  The warp's reads of the stage
// are ordered before it by the __syncwarp() that precedes every call (the
// consumer-release / producer-acquire order of an mbarrier pipeline).
__device__ __forceinline__ void bulk_issue_lane0(int lane, uint32_t dst, uint32_t bar, const void* src, uint32_t bytes,
                                                 uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.eq.s32 p, %0, 0;\n\t"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%2], %4;\n\t"
        "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%1], [%3], %4, [%2], %5;\n\t}" ::"r"(lane),
        "r"(dst), "r"(bar), "l"(src), "r"(bytes), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_lbq_error_word, 0u, code); }

// acc + a.lo * b.lo + a.hi * b.hi: FP16 inputs, exact products, FP32 sums.
__device__ __forceinline__ float fma2_mixed(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ------------------------------------------------------- activation layouts
// Inside a group of 32, x is stored permuted so that each 32-bit word of x
// pairs with the two values one unpack instruction produces.  The 64 bytes of
// a group are four 16-byte chunks; chunk j of 32 consecutive groups are stored
// side by side ([block of 32 groups][chunk][lane]) so that the 32 lanes of a
// warp read 512 contiguous bytes per load.
//
// 4-bit: word j (0..3) of a group's 16 qweight bytes yields the pairs
//   (q_{4j}, q_{4j+2}), (q_{4j+1}, q_{4j+3}), (q_{4j+16}, q_{4j+18}), (q_{4j+17}, q_{4j+19});
// 2-bit: code word v (0..1), shift s (0..3) yields
//   (q_{16v+s}, q_{16v+s+4}) and (q_{16v+s+8}, q_{16v+s+12}).
// Chunk j of a group holds four such pairs of x; natural pairs are
// n_i = (x_{2i}, x_{2i+1}).

__device__ __forceinline__ uint32_t u4w(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// pair of low (sel 0x5410) or high (0x7632) halves of two words
__device__ __forceinline__ uint32_t pair_halves(uint32_t a, uint32_t b, bool high) {
    return prmt(a, b, high ? 0x7632u : 0x5410u);
}

// Permuted chunk j of a group from its 16 natural x pairs n[0..15].
template <int KIND>
__device__ __forceinline__ uint4 permuted_chunk(const uint32_t (&n)[16], int j) {
    uint4 c;
    if (KIND == kW4) {
        // (x_{4j}, x_{4j+2}) (x_{4j+1}, x_{4j+3}) (x_{4j+16}, x_{4j+18}) (x_{4j+17}, x_{4j+19})
        c.x = pair_halves(n[2 * j], n[2 * j + 1], false);
        c.y = pair_halves(n[2 * j], n[2 * j + 1], true);
        c.z = pair_halves(n[8 + 2 * j], n[9 + 2 * j], false);
        c.w = pair_halves(n[8 + 2 * j], n[9 + 2 * j], true);
    } else {
        // word (v, s, pi) = (x_{16v+s+8pi}, x_{16v+s+8pi+4}); chunk j covers (v, s) = (j/2, 2(j%2)..+1)
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int v = j >> 1, s = 2 * (j & 1) + (q >> 1), pi = q & 1;
            const int k1 = 16 * v + s + 8 * pi;
            w[q] = pair_halves(n[k1 >> 1], n[(k1 >> 1) + 2], k1 & 1);
        }
        c = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return c;
}

// uint4 index of chunk j of group g in one activation plane
__device__ __forceinline__ int x_chunk_index(int g, int j) { return ((g >> 5) * 4 + j) * 32 + (g & 31); }

// ------------------------------------------------------ shared-memory plan
//
// [ring: NW * SPW stages][yacc][part][seg][mbarriers][staging of the CTA's problems]
// Staging of one problem: MB permuted activation planes, MB planes of group
// sums, the outlier-channel bitmask, MB rows of gathered outlier activations.

struct FixedPlan {
    int ring, yacc, part, seg, bars, stg, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline FixedPlan fixed_plan(int NW, int stage, int SPW, int MB, int rb_cap) {
    FixedPlan p;
    int off = 0;
    p.ring = off;
    off += NW * SPW * stage;
    p.yacc = off;
    off += rb_cap * kTR * MB * 4;
    p.part = off;
    off += NW * 2 * kTR * MB * 4;
    p.seg = off;
    off += NW * 2 * 4;
    off = round_up(off, 16);
    p.bars = off;
    off += NW * SPW * 8;
    off = round_up(off, 128);
    p.stg = off;
    p.total = off + 128;   // slack for aligning the base to 128 bytes
    return p;
}

__host__ __device__ inline int staging_bytes(int MB, int recs, int OT) {
    const int ng = recs * 32;
    return MB * ng * 64 + MB * ng * 4 + ng * 4 + MB * OT * kOutCols * 2;
}

// Selective refinement pieces of one column that cover rows [n0, n1) of an
// N-row refinement blob, as 16-byte-aligned ranges from the column start: the
// nibble bytes of groups g0 .. g0 + ng - 1 (16 B each), their FP16 scales
// [s_lo, s_lo + ls) and their zero-point bytes [z_lo, z_lo + lz).
struct RefPieces {
    int g0, ng, ln, ls, lz;
    long long s_lo, z_lo;
    __host__ __device__ int bytes() const { return ln + ls + lz; }
};
__host__ __device__ inline RefPieces ref_pieces(long long N, long long n0, long long n1) {
    RefPieces r;
    r.g0 = static_cast<int>(n0 >> 5);
    r.ng = static_cast<int>((n1 - 1) >> 5) - r.g0 + 1;
    r.ln = 16 * r.ng;
    r.s_lo = (N / 2 + 2 * r.g0) & ~15ll;
    r.ls = static_cast<int>(((N / 2 + 2 * (r.g0 + r.ng) + 15) & ~15ll) - r.s_lo);
    r.z_lo = (N / 2 + N / 16 + r.g0 / 2) & ~15ll;
    r.lz = static_cast<int>(((N / 2 + N / 16 + (r.g0 + r.ng - 1) / 2 + 1 + 15) & ~15ll) - r.z_lo);
    return r;
}
// Bytes of the early refinement area of a problem for rows [n0, n1):
// channels (int), x pairs (u32), then the columns' pieces.
__host__ __device__ inline int ref_area_bytes(long long N, long long n0, long long n1, int nsel) {
    return round_up(8 * nsel, 16) + nsel * ref_pieces(N, n0, n1).bytes();
}

// ----------------------------------------------------------- item math
// A dense item is one record; every lane holds its group of the 4 rows.

// 4-bit record, one activation row.  A nibble masked in place is the FP16
// subnormal q * 2^-24 (low nibble) or 16 q * 2^-24 (high nibble); the mixed FMA
// turns it into the exact FP32 product with x.  Per group:
// w.x = s (sum_k q_k x_k - z X_g) = 2^24 s (lo + hi / 16 - z X_g 2^-24);
// the final 2^24 is applied once per output.
__device__ __forceinline__ void w4_record_m1(const uint4 (&q)[kTR], const float (&s)[kTR], const float (&zf)[kTR],
                                             const uint4* xq, float xsz, float (&acc)[kTR]) {
    const uint4 xr[4] = {xq[0], xq[32], xq[64], xq[96]};
    // the 4 rows' 8 accumulation chains are interleaved for instruction-level parallelism
    float lo[kTR], hi[kTR];
#pragma unroll
    for (int r = 0; r < kTR; ++r) lo[r] = hi[r] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
            const uint32_t w = u4w(q[r], j), w8 = w >> 8;
            lo[r] = fma2_mixed(w & 0x000F000Fu, xr[j].x, lo[r]);
            hi[r] = fma2_mixed(w & 0x00F000F0u, xr[j].z, hi[r]);
            lo[r] = fma2_mixed(w8 & 0x000F000Fu, xr[j].y, lo[r]);
            hi[r] = fma2_mixed(w8 & 0x00F000F0u, xr[j].w, hi[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kTR; ++r) {
        const float t = fmaf(-zf[r], xsz, fmaf(hi[r], 0.0625f, lo[r]));
        acc[r] = fmaf(s[r], t, acc[r]);
    }
}

// 4-bit record, MB activation rows: the unpacked words are shared by the rows.
// Every plane is computed, also past the launch's rows (their staged planes are
// zero and their sums are never stored): no branch per plane (measured 3 %
// faster at M = 4).
template <int MB>
__device__ __forceinline__ void w4_record_mb(const uint4 (&q)[kTR], const float (&s)[kTR], const float (&zf)[kTR],
                                             const uint4* xq, int xq_plane, const float* xs24, int xs_plane,
                                             float (&acc)[MB][kTR]) {
    uint32_t u[kTR][16];
#pragma unroll
    for (int r = 0; r < kTR; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t w = u4w(q[r], j), w8 = w >> 8;
            u[r][4 * j + 0] = w & 0x000F000Fu;
            u[r][4 * j + 1] = w8 & 0x000F000Fu;
            u[r][4 * j + 2] = w & 0x00F000F0u;
            u[r][4 * j + 3] = w8 & 0x00F000F0u;
        }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        {
            const uint4* xp = xq + m * xq_plane;
            const uint4 xr[4] = {xp[0], xp[32], xp[64], xp[96]};
            const float xsz = xs24[m * xs_plane];
            float lo[kTR], hi[kTR];
#pragma unroll
            for (int r = 0; r < kTR; ++r) lo[r] = hi[r] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int r = 0; r < kTR; ++r) {
                    lo[r] = fma2_mixed(u[r][4 * j + 0], xr[j].x, lo[r]);
                    hi[r] = fma2_mixed(u[r][4 * j + 2], xr[j].z, hi[r]);
                    lo[r] = fma2_mixed(u[r][4 * j + 1], xr[j].y, lo[r]);
                    hi[r] = fma2_mixed(u[r][4 * j + 3], xr[j].w, hi[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                const float t = fmaf(-zf[r], xsz, fmaf(hi[r], 0.0625f, lo[r]));
                acc[m][r] = fmaf(s[r], t, acc[m][r]);
            }
        }
    }
}

// 2-bit record: four codes -> PRMT selector (c, c+4 per code) -> two FP16
// codebook pairs; w.x = S sum_k C[q_k] x_k + Z X_g.
__device__ __forceinline__ void w2_record(const uint2 (&c)[kTR], const float (&S)[kTR], const float (&Z)[kTR],
                                          const uint4* xq, float xs, uint32_t lut_lo, uint32_t lut_hi,
                                          float (&acc)[kTR]) {
    const uint4 xr[4] = {xq[0], xq[32], xq[64], xq[96]};
    // the 4 rows' 8 accumulation chains are interleaved for instruction-level parallelism
    float d0[kTR], d1[kTR];
#pragma unroll
    for (int r = 0; r < kTR; ++r) d0[r] = d1[r] = 0.f;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
#pragma unroll
        for (int sh = 0; sh < 4; ++sh) {
            const int mw = (v * 4 + sh) * 2;                       // word of the group's 64 x bytes
            const uint32_t xa = u4w(xr[mw >> 2], mw & 3), xb = u4w(xr[(mw + 1) >> 2], (mw + 1) & 3);
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                const uint32_t w = v ? c[r].y : c[r].x;
                const uint32_t t = (w >> (2 * sh)) & 0x03030303u;
                const uint32_t sel = t * 0x11u + 0x40404040u;     // nibbles (c, c + 4) per code
                d0[r] = fma2_mixed(prmt(lut_lo, lut_hi, sel), xa, d0[r]);
                d1[r] = fma2_mixed(prmt(lut_lo, lut_hi, sel >> 16), xb, d1[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kTR; ++r) acc[r] = fmaf(S[r], d0[r] + d1[r], fmaf(Z[r], xs, acc[r]));
}

// 2-bit record, MB activation rows: the codebook pairs of the 4 rows are
// decoded once (PRMT as above) and shared by the rows' FMAs; every plane is
// computed, as for 4-bit.
template <int MB>
__device__ __forceinline__ void w2_record_mb(const uint2 (&c)[kTR], const float (&S)[kTR], const float (&Z)[kTR],
                                             const uint4* xq, int xq_plane, const float* xs, int xs_plane,
                                             uint32_t lut_lo, uint32_t lut_hi, float (&acc)[MB][kTR]) {
    uint32_t p[kTR][16];   // pair (v * 4 + sh) * 2 + h: codes of word v, shift sh, half h
#pragma unroll
    for (int r = 0; r < kTR; ++r)
#pragma unroll
        for (int v = 0; v < 2; ++v)
#pragma unroll
            for (int sh = 0; sh < 4; ++sh) {
                const uint32_t t = ((v ? c[r].y : c[r].x) >> (2 * sh)) & 0x03030303u;
                const uint32_t sel = t * 0x11u + 0x40404040u;
                p[r][(v * 4 + sh) * 2] = prmt(lut_lo, lut_hi, sel);
                p[r][(v * 4 + sh) * 2 + 1] = prmt(lut_lo, lut_hi, sel >> 16);
            }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        {
            const uint4* xp = xq + m * xq_plane;
            const uint4 xr[4] = {xp[0], xp[32], xp[64], xp[96]};
            float d0[kTR], d1[kTR];
#pragma unroll
            for (int r = 0; r < kTR; ++r) d0[r] = d1[r] = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int mw = 2 * w;                              // word of the group's 64 x bytes
                const uint32_t xa = u4w(xr[mw >> 2], mw & 3), xb = u4w(xr[(mw + 1) >> 2], (mw + 1) & 3);
#pragma unroll
                for (int r = 0; r < kTR; ++r) {
                    d0[r] = fma2_mixed(p[r][2 * w], xa, d0[r]);
                    d1[r] = fma2_mixed(p[r][2 * w + 1], xb, d1[r]);
                }
            }
            const float xsm = xs[m * xs_plane];
#pragma unroll
            for (int r = 0; r < kTR; ++r) acc[m][r] = fmaf(S[r], d0[r] + d1[r], fmaf(Z[r], xsm, acc[m][r]));
        }
    }
}

// One outlier record: lane owns outlier columns [lane*8, +8) of the record's 256
// for the 4 rows; xo + m * xo_plane holds x[idx] of activation row m.  `unit`
// converts to the unit of the dense accumulator (2^-24 for 4-bit, 1 for 2-bit).
template <int MB>
__device__ __forceinline__ void outlier_record(const uint4 (&v)[kTR], const __half* xo, int xo_plane, int mrows,
                                               int lane, float unit, float (&acc)[MB][kTR]) {
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        if (m < mrows) {
            const uint4 xv = reinterpret_cast<const uint4*>(xo + m * xo_plane)[lane];
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                float a0 = fma2_mixed(v[r].x, xv.x, 0.f);
                float a1 = fma2_mixed(v[r].y, xv.y, 0.f);
                a0 = fma2_mixed(v[r].z, xv.z, a0);
                a1 = fma2_mixed(v[r].w, xv.w, a1);
                acc[m][r] = fmaf(a0 + a1, unit, acc[m][r]);
            }
        }
    }
}

// Sum acc[0..3] over the 32 lanes; lane 8r ends with row r's total.
__device__ __forceinline__ float reduce_rows4(const float (&acc)[4], int lane) {
    const bool up = lane & 16;
    float keep0 = up ? acc[2] : acc[0];
    float keep1 = up ? acc[3] : acc[1];
    const float send0 = up ? acc[0] : acc[2];
    const float send1 = up ? acc[1] : acc[3];
    keep0 += __shfl_xor_sync(0xffffffffu, send0, 16);
    keep1 += __shfl_xor_sync(0xffffffffu, send1, 16);
    const bool b3 = lane & 8;
    float m = b3 ? keep1 : keep0;
    const float u = b3 ? keep0 : keep1;
    m += __shfl_xor_sync(0xffffffffu, u, 8);
    m += __shfl_xor_sync(0xffffffffu, m, 4);
    m += __shfl_xor_sync(0xffffffffu, m, 2);
    m += __shfl_xor_sync(0xffffffffu, m, 1);
    return m;
}

// ------------------------------------------------------------------ kernel

__device__ __forceinline__ int unit_end(const GroupArgs& a, int q) { return q + 1 < a.count ? a.p[q + 1].ub : a.nunits; }

// The 8-warp M = 1 variants are built for two resident CTAs per SM (<= 128
// registers a thread), so that a dependent launch's CTAs can start beside them.
template <int KIND, int MB, int NW, int RPI>
__global__ void __launch_bounds__(NW * 32, (MB == 1 && NW == 8) ? 2 : 1) lbq_gemv_kernel(const __grid_constant__ GroupArgs a) {
    using RC = Rec<KIND>;
    constexpr int kStage = RC::template stage<RPI>();
    constexpr int kThreads = NW * 32;
    constexpr float kUnit = KIND == kW4 ? 5.9604644775390625e-8f : 1.f;   // 2^-24 for the 4-bit products
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // align by offsetting the shared array itself, so the compiler keeps the
    // shared address space (LDS with immediate offsets, no generic addressing)
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    // M = 1 kernels always run 2 stages per warp (the host plans exactly that)
    const int SPW = MB == 1 ? kStagesM1 : a.SPW;
    const FixedPlan P = fixed_plan(NW, kStage, SPW, MB, a.rb_cap);
    float* yacc = reinterpret_cast<float*>(smem + P.yacc);
    float* part = reinterpret_cast<float*>(smem + P.part);
    int* seg = reinterpret_cast<int*>(smem + P.seg);
    uint8_t* stg = smem + P.stg;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mrows = a.mrows;
    const int u0 = a.cta_ub[blockIdx.x], u1 = a.cta_ub[blockIdx.x + 1];
    const int R = u1 - u0;

    // problems this CTA touches: qf .. qf + np - 1; its items (records and
    // outlier records of its row blocks, in memory order).  Lane l of every warp
    // reads problem l's scalars (at most 32 problems), so the launch parameters
    // are fetched in one round instead of a chain of dependent reads (measured:
    // ~1.8 us of prologue before), and the loops over problems become ballots and
    // warp scans.
    const bool lp = lane < a.count;
    const int p_ub = lp ? a.p[lane].ub : INT_MAX;
    const int p_end = lp ? (lane + 1 < a.count ? a.p[lane + 1].ub : a.nunits) : INT_MAX;
    const int p_recs = lp ? a.p[lane].recs : 0, p_OT = lp ? a.p[lane].OT : 0;
    const int qf = __popc(__ballot_sync(0xffffffffu, p_ub <= u0)) - 1;   // ub ascending, ub[0] = 0
    const bool in_cta = R > 0 && lp && lane >= qf && p_ub < u1;
    const int np = __popc(__ballot_sync(0xffffffffu, in_cta));
    const int p_tpr = (p_recs + RPI - 1) / RPI + p_OT;                    // items per row block
    const int p_items = in_cta ? (min(u1, p_end) - max(u0, p_ub)) * p_tpr : 0;
    const int p_stg = in_cta ? staging_bytes(MB, p_recs, p_OT) : 0;
    int items_incl = p_items, stg_incl = p_stg;                           // inclusive warp scans
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int vi = __shfl_up_sync(0xffffffffu, items_incl, d), vs = __shfl_up_sync(0xffffffffu, stg_incl, d);
        if (lane >= d) {
            items_incl += vi;
            stg_incl += vs;
        }
    }
    const int n_items = __shfl_sync(0xffffffffu, items_incl, 31);
    // this warp's contiguous share of the items, and where it starts
    const int ib = static_cast<int>((static_cast<long long>(warp) * n_items) / NW);
    const int ie = static_cast<int>((static_cast<long long>(warp + 1) * n_items) / NW);
    const int my_items = ie - ib;
    int s_q = qf, s_stg = 0, s_u = u0, s_kk = 0;
    if (my_items > 0) {
        // the problem whose items hold ib: the first lane whose inclusive count exceeds ib
        const int sl = __ffs(__ballot_sync(0xffffffffu, in_cta && items_incl > ib)) - 1;
        const int before = __shfl_sync(0xffffffffu, items_incl - p_items, sl);
        const int tpr = __shfl_sync(0xffffffffu, p_tpr, sl), lo = __shfl_sync(0xffffffffu, max(u0, p_ub), sl);
        s_q = sl;
        s_stg = __shfl_sync(0xffffffffu, stg_incl - p_stg, sl);
        const int j = ib - before;
        s_u = lo + j / tpr;
        s_kk = j - (j / tpr) * tpr;
    }
    uint64_t* my_bars = reinterpret_cast<uint64_t*>(smem + P.bars) + warp * SPW;
    uint8_t* my_ring = smem + P.ring + warp * SPW * kStage;

    // issue pointer (warp-uniform; only lane 0 executes the copies): problem,
    // row block, item, source address, slot
    int i_q = s_q, i_u = s_u, i_kk = s_kk, i_slot = 0;
    int i_recs = a.p[s_q].recs, i_di = (i_recs + RPI - 1) / RPI, i_TPR = i_di + a.p[s_q].OT;
    int i_uend = min(u1, unit_end(a, s_q));
    int i_last = a.p[s_q].out_last;
    const uint8_t* i_src = a.p[s_q].area + static_cast<long long>(s_u - a.p[s_q].ub) * a.p[s_q].rb_bytes +
                           (s_kk < i_di ? static_cast<long long>(s_kk) * RPI * RC::kBytes
                                        : static_cast<long long>(i_recs) * RC::kBytes +
                                              static_cast<long long>(s_kk - i_di) * kOutRecBytes);
    const uint64_t policy = policy_evict_first();
    const uint32_t ring_u32 = smem_u32(my_ring), bars_u32 = smem_u32(my_bars);
    auto issue_next = [&](bool more) {
        const uint32_t bytes = i_kk < i_di         ? static_cast<uint32_t>(min(RPI, i_recs - i_kk * RPI) * RC::kBytes)
                               : i_kk + 1 == i_TPR ? static_cast<uint32_t>(i_last)
                                                   : static_cast<uint32_t>(kOutRecBytes);
        bulk_issue_lane0(more ? lane : 1, ring_u32 + i_slot * kStage, bars_u32 + i_slot * 8, i_src, bytes, policy);
        i_src += bytes;   // the row blocks of a problem are contiguous
        if (++i_kk == i_TPR) {
            i_kk = 0;
            if (++i_u == i_uend && ++i_q < a.count) {
                // next problem, entered at its first row block
                i_recs = a.p[i_q].recs;
                i_di = (i_recs + RPI - 1) / RPI;
                i_TPR = i_di + a.p[i_q].OT;
                i_last = a.p[i_q].out_last;
                i_uend = min(u1, unit_end(a, i_q));
                i_src = a.p[i_q].area;
            }
        }
        if (++i_slot == SPW) i_slot = 0;
    };

    // barriers, then start the weight stream before waiting on the previous grid
    if (lane == 0) {
        for (int s = 0; s < SPW; ++s) mbar_init(my_bars + s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    {
        const int pre = my_items < SPW ? my_items : SPW;
        for (int t = 0; t < pre; ++t) issue_next(true);
    }
    // blob header of problem blockIdx.x: loaded now, compared after the main
    // loop, so the check never delays this CTA's prologue
    uint4 hdr0 = make_uint4(0u, 0u, 0u, 0u), hdr1 = hdr0, hdr2 = hdr0, rhdr0 = hdr0, rhdr1 = hdr0;
    const bool check_hdr = static_cast<int>(blockIdx.x) < a.count && tid == 0;
    if (check_hdr) {
        const uint4* h = reinterpret_cast<const uint4*>(a.p[blockIdx.x].blob);
        hdr0 = h[0];
        hdr1 = h[1];
        hdr2 = h[2];
    }
    // and its refinement blob's header (magic, version, N, K)
    const bool check_rhdr = MB == 1 && static_cast<int>(blockIdx.x) < a.count && tid == 32 && a.p[blockIdx.x].nsel > 0;
    if (check_rhdr) {
        const uint4* h = reinterpret_cast<const uint4*>(a.p[blockIdx.x].rblob);
        rhdr0 = h[0];
        rhdr1 = h[1];
    }
    // outlier-channel bitmasks and the row accumulators (no dependence on the previous grid)
    bool any_out = false;
    {
        int off = 0;
        for (int j = 0, q = qf; j < np; ++j, ++q) {
            const int ng = a.p[q].recs * 32;
            if (a.p[q].n_out > 0) {
                any_out = true;
                uint32_t* om = reinterpret_cast<uint32_t*>(stg + off + MB * ng * 68);
                for (int i = tid; i < ng; i += kThreads) om[i] = 0u;
            }
            off += staging_bytes(MB, a.p[q].recs, a.p[q].OT);
        }
    }
    for (int i = tid; i < R * kTR * MB; i += kThreads) yacc[i] = 0.f;
    pdl_trigger();
    if (any_out) {
        __syncthreads();
        int off = 0;
        for (int j = 0, q = qf; j < np; ++j, ++q) {
            const int ng = a.p[q].recs * 32;
            uint32_t* om = reinterpret_cast<uint32_t*>(stg + off + MB * ng * 68);
            const int n_out = a.p[q].n_out;
            const int32_t* idx = a.p[q].idx;
            const long long K = a.p[q].K;
            for (int i = tid; i < n_out; i += kThreads) {
                const int k = idx[i];
                if (k >= 0 && k < K)
                    atomicOr(&om[k >> 5], 1u << (k & 31));
                else
                    record_error(LBQ_ERR_OUTLIER_IDX);   // corrupted blob: never index outside x
            }
            off += staging_bytes(MB, a.p[q].recs, a.p[q].OT);
        }
    }
    __syncthreads();
    pdl_wait();

    // selective refinement, early staging (M = 1): the area after the CTA's
    // staging holds, per refined problem, its chosen channels, their x pairs and
    // the chosen columns' pieces covering the CTA's rows.  The channels are copied
    // now (asynchronously, while x is staged), the pieces right before the main
    // loop, so that they land while the weights stream.
    uint8_t* rarea = nullptr;
    if (MB == 1 && a.rearly && R > 0) {
        int off = 0;
        for (int j = 0, q = qf; j < np; ++j, ++q) off += staging_bytes(MB, a.p[q].recs, a.p[q].OT);
        rarea = stg + off;
        int aoff = 0;
        for (int q = qf; q < a.count && a.p[q].ub < u1; ++q) {
            const ProbArg& pa = a.p[q];
            const int lo = max(u0, pa.ub), hi = min(u1, unit_end(a, q));
            const long long n0 = static_cast<long long>(lo - pa.ub) * kTR;
            const long long n1 = min(pa.N, static_cast<long long>(hi - pa.ub) * kTR);
            if (pa.nsel <= 0 || n1 <= n0) continue;
            for (int jj = tid; jj < pa.nsel; jj += kThreads)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(rarea + aoff + 4 * jj)),
                             "l"(pa.ridx + jj)
                             : "memory");
            aoff += ref_area_bytes(pa.N, n0, n1, pa.nsel);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // stage x of every problem: a thread takes whole groups (four 16-byte loads),
    // zeroes outlier channels, writes the permuted chunks and the group sum X~_g
    // (times kUnit); then x[idx] (the unmasked values) for the outlier records
    {
        int off = 0;
        for (int j = 0, q = qf; j < np; ++j, ++q) {
            const ProbArg& pa = a.p[q];
            const int ng = pa.recs * 32;
            uint4* xs = reinterpret_cast<uint4*>(stg + off);
            float* xsum = reinterpret_cast<float*>(stg + off + MB * ng * 64);
            const uint32_t* om = reinterpret_cast<const uint32_t*>(stg + off + MB * ng * 68);
            __half* xo = reinterpret_cast<__half*>(stg + off + MB * ng * 68 + ng * 4);
            const int xq_plane = ng * 4;
            for (int base = tid; base < MB * ng; base += kThreads * 2) {
                uint4 raw[2][4];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int i = base + b * kThreads;
                    const int m = i / ng, g = i - m * ng;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        raw[b][c] = make_uint4(0u, 0u, 0u, 0u);
                        if (i < MB * ng && m < mrows && g * 32 < pa.K)
                            raw[b][c] = *reinterpret_cast<const uint4*>(pa.x + m * pa.ldx + g * 32 + c * 8);
                    }
                }
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int i = base + b * kThreads;
                    if (i < MB * ng) {
                        const int m = i / ng, g = i - m * ng;
                        uint32_t n[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            n[4 * c + 0] = raw[b][c].x;
                            n[4 * c + 1] = raw[b][c].y;
                            n[4 * c + 2] = raw[b][c].z;
                            n[4 * c + 3] = raw[b][c].w;
                        }
                        const uint32_t omw = pa.n_out > 0 ? om[g] : 0u;
                        if (omw) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const uint32_t keep = ((omw >> (2 * e)) & 1u ? 0xFFFF0000u : 0xFFFFFFFFu) &
                                                      ((omw >> (2 * e + 1)) & 1u ? 0x0000FFFFu : 0xFFFFFFFFu);
                                n[e] &= keep;
                            }
                        }
                        float s0 = 0.f, s1 = 0.f;
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            s0 = fma2_mixed(n[e], 0x3C003C00u, s0);         // + x_{2e} + x_{2e+1}
                            s1 = fma2_mixed(n[e + 1], 0x3C003C00u, s1);
                        }
                        // 4-bit: the zero point arrives as z * 2^-24 (even groups) or
                        // 16 z * 2^-24 (odd groups, high nibble), so odd sums are staged / 16
                        xsum[i] = (KIND == kW4 && (g & 1)) ? (s0 + s1) * 0.0625f : (s0 + s1);
                        uint4* dst = xs + m * xq_plane;
#pragma unroll
                        for (int c = 0; c < 4; ++c) dst[x_chunk_index(g, c)] = permuted_chunk<KIND>(n, c);
                    }
                }
            }
            const int xo_plane = pa.OT * kOutCols;
            for (int i = tid; i < MB * xo_plane; i += kThreads) {
                const int m = i / xo_plane, jj = i - m * xo_plane;
                __half v = __float2half(0.f);
                if (jj < pa.n_out && m < mrows) {
                    const int k = pa.idx[jj];
                    if (k >= 0 && k < pa.K) v = pa.x[m * pa.ldx + k];
                }
                xo[i] = v;
            }
            off += staging_bytes(MB, pa.recs, pa.OT);
        }
    }
    __syncthreads();
    if (rarea) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // every thread's channel copies have landed
        int aoff = 0;
        for (int q = qf; q < a.count && a.p[q].ub < u1; ++q) {
            const ProbArg& pa = a.p[q];
            const int lo = max(u0, pa.ub), hi = min(u1, unit_end(a, q));
            const long long n0 = static_cast<long long>(lo - pa.ub) * kTR;
            const long long n1 = min(pa.N, static_cast<long long>(hi - pa.ub) * kTR);
            if (pa.nsel <= 0 || n1 <= n0) continue;
            const RefPieces rp = ref_pieces(pa.N, n0, n1);
            const int lc = rp.bytes(), pieces = lc / 16;
            const int* rs = reinterpret_cast<const int*>(rarea + aoff);
            uint8_t* raw = rarea + aoff + round_up(8 * pa.nsel, 16);
            const uint8_t* cols = pa.rblob + lbq::kRefineHeader;
            for (int pi = tid; pi < pa.nsel * pieces; pi += kThreads) {
                const int jj = pi / pieces, k = pi - jj * pieces;
                const int c = rs[jj] >= 0 && rs[jj] < pa.K ? rs[jj] : 0;   // a bad channel is reported later
                const uint8_t* col = cols + static_cast<long long>(c) * pa.rcb;
                const uint8_t* src = k * 16 < rp.ln           ? col + 16 * rp.g0 + 16 * k
                                     : k * 16 < rp.ln + rp.ls ? col + rp.s_lo + (16 * k - rp.ln)
                                                              : col + rp.z_lo + (16 * k - rp.ln - rp.ls);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(raw + jj * lc + 16 * k)),
                             "l"(src)
                             : "memory");
            }
            // the 4-byte pair of x holding x[c]
            for (int jj = tid; jj < pa.nsel; jj += kThreads) {
                const int c = rs[jj] >= 0 && rs[jj] < pa.K ? rs[jj] : 0;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(rarea + aoff + 4 * pa.nsel + 4 * jj)),
                             "l"(pa.x + (c & ~1))
                             : "memory");
            }
            aoff += ref_area_bytes(pa.N, n0, n1, pa.nsel);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // main loop: this warp's items through its ring, one segment (a run of
    // items of one row block: its dense records, then its outlier records) at a time
    bool ok = true;
    int c_q = s_q, c_u = s_u, c_kk = s_kk, c_slot = 0, c_stg = s_stg;
    uint32_t c_phase = 0;
    int c_recs = a.p[s_q].recs, c_OT = a.p[s_q].OT, c_di = (c_recs + RPI - 1) / RPI, c_TPR = c_di + c_OT;
    int c_uend = min(u1, unit_end(a, s_q));
    int c_out_last = a.p[s_q].out_last;
    const int first_lu = my_items > 0 ? s_u - u0 : -1;
    if (lane == 0) {
        seg[2 * warp] = first_lu;
        seg[2 * warp + 1] = -1;
    }
    // lane 0 of a record's zero byte holds group 2m in the low nibble, lane 1
    // group 2m+1 in the high one; masked in place it is the FP16 subnormal
    // z * 2^-24 or 16 z * 2^-24 (the group sums of odd groups are staged / 16)
    const uint32_t zmask = (lane & 1) ? 0xF0u : 0x0Fu;
    float acc[MB][kTR];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int r = 0; r < kTR; ++r) acc[m][r] = 0.f;
    int t = 0;
    // one step of the ring: wait for the stage (warp-uniform), run `body` on it
    // after the refill of the stage has been handed to lane 0's copy engine
    auto next_stage = [&](auto&& load, auto&& body) -> bool {
        uint64_t* bar = my_bars + c_slot;
        if (!__all_sync(0xffffffffu, mbar_try_wait(bar, c_phase)) &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(bar, c_phase, kWaitLimitNs)))
            return false;                                  // a lane timed out: the warp aborts
        const uint8_t* st = my_ring + c_slot * kStage;
        load(st);                                          // the item into registers
        __syncwarp();
        issue_next(t + SPW < my_items);                    // hand the stage back
        c_slot = c_slot + 1 == SPW ? 0 : c_slot + 1;
        c_phase ^= c_slot == 0 ? 1u : 0u;
        body();
        return true;
    };
    while (t < my_items && ok) {
        const int seg_n = min(my_items - t, c_TPR - c_kk);
        const int nd = max(0, min(seg_n, c_di - c_kk));        // dense items of the segment
        const int ng = c_recs * 32;
        const uint4* xq = reinterpret_cast<const uint4*>(stg + c_stg) + c_kk * RPI * 128 + lane;
        const float* xsg = reinterpret_cast<const float*>(stg + c_stg + MB * ng * 64) + c_kk * RPI * 32 + lane;
        const __half* xo = reinterpret_cast<const __half*>(stg + c_stg + MB * ng * 68 + ng * 4) +
                           max(0, c_kk - c_di) * kOutCols;
        const int t_end = t + seg_n, t_dense = t + nd;
        uint4 q4[kTR];
        float f1[kTR], f2[kTR];
        // dense items: RPI consecutive records (the last item of a row block may
        // hold fewer); the stage is handed back once its last record is in
        // registers, the records before it are computed while it is held
        for (int dk = c_kk; t < t_dense; ++t, ++dk) {
            const int nrec = min(RPI, c_recs - RPI * dk);
            if constexpr (KIND == kW4) {
                auto load_rec = [&](const uint8_t* st) {
#pragma unroll
                    for (int r = 0; r < kTR; ++r) {
                        q4[r] = reinterpret_cast<const uint4*>(st)[r * 32 + lane];
                        f1[r] = __half2float(reinterpret_cast<const __half*>(st + RC::kOff1)[r * 32 + lane]);
                        const uint32_t zb = st[RC::kOff2 + r * 16 + (lane >> 1)] & zmask;
                        f2[r] = __half2float(__ushort_as_half(static_cast<unsigned short>(zb)));
                    }
                };
                auto compute = [&](const uint4* xqq, const float* xss) {
                    if constexpr (MB == 1)
                        w4_record_m1(q4, f1, f2, xqq, *xss, acc[0]);
                    else
                        w4_record_mb<MB>(q4, f1, f2, xqq, ng * 4, xss, ng, acc);
                };
                ok = next_stage(
                    [&](const uint8_t* st) {
                        load_rec(st);
#pragma unroll
                        for (int j = 1; j < RPI; ++j)
                            if (j < nrec) {
                                compute(xq + 128 * (j - 1), xsg + 32 * (j - 1));
                                load_rec(st + j * RC::kBytes);
                            }
                    },
                    [&]() { compute(xq + 128 * (nrec - 1), xsg + 32 * (nrec - 1)); });
            } else {
                uint2 q2[kTR];
                auto load_rec = [&](const uint8_t* st) {
#pragma unroll
                    for (int r = 0; r < kTR; ++r) {
                        q2[r] = reinterpret_cast<const uint2*>(st)[r * 32 + lane];
                        f1[r] = __half2float(reinterpret_cast<const __half*>(st + RC::kOff1)[r * 32 + lane]);
                        f2[r] = __half2float(reinterpret_cast<const __half*>(st + RC::kOff2)[r * 32 + lane]);
                    }
                };
                auto compute = [&](const uint4* xqq, const float* xss) {
                    if constexpr (MB == 1)
                        w2_record(q2, f1, f2, xqq, *xss, a.lut_lo, a.lut_hi, acc[0]);
                    else
                        w2_record_mb<MB>(q2, f1, f2, xqq, ng * 4, xss, ng, a.lut_lo, a.lut_hi, acc);
                };
                ok = next_stage(
                    [&](const uint8_t* st) {
                        load_rec(st);
#pragma unroll
                        for (int j = 1; j < RPI; ++j)
                            if (j < nrec) {
                                compute(xq + 128 * (j - 1), xsg + 32 * (j - 1));
                                load_rec(st + j * RC::kBytes);
                            }
                    },
                    [&]() { compute(xq + 128 * (nrec - 1), xsg + 32 * (nrec - 1)); });
            }
            if (!ok) break;
            xq += 128 * nrec;
            xsg += 32 * nrec;
        }
        // outlier records: 256 columns each, the last one trimmed (its rows are
        // `cols` wide); a lane owns 8 columns, lanes past the width read zeros
        for (int o = max(0, c_kk - c_di); ok && t < t_end; ++t, ++o) {
            const int cols = o + 1 == c_OT ? c_out_last / 8 : kOutCols;
            ok = next_stage(
                [&](const uint8_t* st) {
                    const bool mine = lane * 8 < cols;
#pragma unroll
                    for (int r = 0; r < kTR; ++r)
                        q4[r] = mine ? *reinterpret_cast<const uint4*>(st + r * cols * 2 + lane * 16)
                                     : make_uint4(0u, 0u, 0u, 0u);
                },
                [&]() { outlier_record<MB>(q4, xo, c_OT * kOutCols, mrows, lane, kUnit, acc); });
            if (!ok) break;
            xo += kOutCols;
        }
        if (!ok) break;
        // end of a segment: reduce over lanes and park the row partials
        const bool last = t == my_items;
        const int lu = c_u - u0;
        const int pslot = (lu == first_lu) ? 0 : (last ? 1 : -1);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            if (m < mrows) {
                const float tot = reduce_rows4(acc[m], lane);
                if ((lane & 7) == 0) {
                    const int r = lane >> 3;
                    if (pslot < 0)
                        yacc[(lu * kTR + r) * MB + m] = tot;             // row block owned by this warp alone
                    else
                        part[((warp * 2 + pslot) * kTR + r) * MB + m] = tot;
                }
            }
#pragma unroll
            for (int r = 0; r < kTR; ++r) acc[m][r] = 0.f;
        }
        if (last && lane == 0 && lu != first_lu) seg[2 * warp + 1] = lu;
        c_kk += seg_n;
        if (c_kk == c_TPR && !last) {
            c_kk = 0;
            if (++c_u == c_uend) {
                c_stg += staging_bytes(MB, c_recs, c_OT);
                ++c_q;
                c_recs = a.p[c_q].recs;
                c_OT = a.p[c_q].OT;
                c_out_last = a.p[c_q].out_last;
                c_di = (c_recs + RPI - 1) / RPI;
                c_TPR = c_di + c_OT;
                c_uend = min(u1, unit_end(a, c_q));
            }
        }
    }
    if (!ok) {
        if (lane == 0) {
            record_error(LBQ_ERR_TIMEOUT);
            // drain the copies this warp still has in flight before its shared memory goes away
            const int outstanding = (my_items - t) < SPW ? (my_items - t) : SPW;
            for (int u = 0; u < outstanding; ++u) {
                const int slot = (c_slot + u) % SPW;
                const uint32_t ph = (slot >= c_slot) ? c_phase : (c_phase ^ 1u);
                mbar_wait_bounded(my_bars + slot, ph, kWaitLimitNs / 8);
            }
        }
        __syncwarp();
    }
    __syncthreads();

    // selective refinement (M = 1; StrataFlux section 3, Eq. 2): the corrections
    // sum_j x[idx_j] C[n, idx_j] of the CTA's rows, in FP32.  The chosen columns'
    // pieces that cover the CTA's rows (nibble bytes of its 32-row groups, their
    // scales and zero points) are in the early area (staged while the weights
    // streamed), or, when that did not fit in shared memory, are copied now into
    // the free stage ring, all in flight at once (the selection kernel before
    // this one prefetched them into L2), in batches that fit.  A thread then
    // takes one 32-bit nibble word (8 rows of a group) and one slice of the
    // columns (column j in slice j % WS, ascending); the slices' partial rows are
    // added in slice order into rfin (a fixed order), which the combine below
    // adds to y.
    // ring: [rfin: RR floats][channels, x values: batch][word partials][columns]
    const int RR = R * kTR;
    float* rfin = reinterpret_cast<float*>(smem + P.ring);
    const int fin_bytes = round_up(RR * 4, 16);
    int* rsel_b = reinterpret_cast<int*>(smem + P.ring + fin_bytes);
    float* rx_b = reinterpret_cast<float*>(rsel_b + kRefineBatchMax);
    float* wpart = rx_b + kRefineBatchMax;
    const int fixed_bytes = fin_bytes + 8 * kRefineBatchMax;
    bool refined = false;
    if (MB == 1 && R > 0)
        for (int q = qf; q < a.count && a.p[q].ub < u1; ++q) refined = refined || a.p[q].nsel > 0;
    if (refined) {
        if (rarea) asm volatile("cp.async.wait_group 0;" ::: "memory");   // this thread's early pieces
        for (int i = tid; i < RR; i += kThreads) rfin[i] = 0.f;
        int aoff = 0;
        for (int q = qf; q < a.count && a.p[q].ub < u1; ++q) {
            const ProbArg& pa = a.p[q];
            if (pa.nsel <= 0) continue;
            const int lo = max(u0, pa.ub), hi = min(u1, unit_end(a, q));
            const long long n0 = static_cast<long long>(lo - pa.ub) * kTR;
            const long long n1 = min(pa.N, static_cast<long long>(hi - pa.ub) * kTR);
            if (n1 <= n0) continue;
            const int rl0 = (lo - u0) * kTR;                 // CTA-local row of n0
            const RefPieces rp = ref_pieces(pa.N, n0, n1);
            const int g0 = rp.g0, ng = rp.ng, ln = rp.ln, ls = rp.ls;
            const int lc = rp.bytes(), pieces = lc / 16;
            // words of the CTA's groups; word threads and column slices
            const int nw = 4 * ng, WT = nw < kThreads ? nw : kThreads, WS = kThreads / WT;
            const int wt = tid % WT, ws = tid / WT;
            const int wbytes = 32 * WS * nw;                  // 8 row partials per (slice, word)
            __syncthreads();   // the previous problem's partials have been read (and the early pieces landed)
            for (int i = tid; i < 8 * WS * nw; i += kThreads) wpart[i] = 0.f;
            // one batch of columns j0 .. j0 + nb - 1: pieces at raw, x values at rx
            auto accumulate = [&](const uint8_t* raw, const float* rx, int j0, int nb) {
                if (ws >= WS) return;
                for (int wi = wt; wi < nw; wi += WT) {
                    const int g = wi >> 2, w = wi & 3;
                    const int so = static_cast<int>(pa.N / 2 + 2 * (g0 + g) - rp.s_lo);
                    const int zo = static_cast<int>(pa.N / 2 + pa.N / 16 + (g0 + g) / 2 - rp.z_lo);
                    const int zsh = ((g0 + g) & 1) ? 4 : 0;
                    float* wp = wpart + (ws * nw + wi) * 8;
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = wp[e];
                    for (int jj = (ws - j0 % WS + WS) % WS; jj < nb; jj += WS) {   // (j0 + jj) % WS == ws
                        const uint8_t* cp = raw + jj * lc;
                        const uint32_t word = *reinterpret_cast<const uint32_t*>(cp + 16 * g + 4 * w);
                        const float sc = __half2float(*reinterpret_cast<const __half*>(cp + ln + so));
                        const float zf = static_cast<float>((cp[ln + ls + zo] >> zsh) & 15u);
                        const float xs = rx[jj];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            // rows 32 g + 4 w + b (low nibble), 32 g + 16 + 4 w + b (high);
                            // (q - z) s is exact in FP32
                            acc[b] = fmaf((static_cast<float>((word >> (8 * b)) & 15u) - zf) * sc, xs, acc[b]);
                            acc[4 + b] =
                                fmaf((static_cast<float>((word >> (8 * b + 4)) & 15u) - zf) * sc, xs, acc[4 + b]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) wp[e] = acc[e];
                }
            };
            if (rarea) {
                // early area: channels, x pairs -> x values in place, pieces
                int* rs = reinterpret_cast<int*>(rarea + aoff);
                uint32_t* xp = reinterpret_cast<uint32_t*>(rarea + aoff + 4 * pa.nsel);
                for (int jj = tid; jj < pa.nsel; jj += kThreads) {
                    const int c = rs[jj];
                    float xv = 0.f;
                    if (c >= 0 && c < pa.K)
                        xv = __half2float(__ushort_as_half(static_cast<unsigned short>(xp[jj] >> (16 * (c & 1)))));
                    else
                        record_error(LBQ_ERR_VALUE);   // skipped: its x counts as 0
                    reinterpret_cast<float*>(xp)[jj] = xv;
                }
                __syncthreads();
                accumulate(rarea + aoff + round_up(8 * pa.nsel, 16), reinterpret_cast<const float*>(xp), 0, pa.nsel);
                aoff += ref_area_bytes(pa.N, n0, n1, pa.nsel);
            } else {
                uint8_t* raw = smem + P.ring + fixed_bytes + wbytes;
                int per = (P.yacc - P.ring - fixed_bytes - wbytes) / lc;
                per = per < kRefineBatchMax ? per : kRefineBatchMax;
                if (per < 1) {   // row ranges this long are not planned with a refinement
                    if (tid == 0) record_error(LBQ_ERR_SHAPE);
                    break;
                }
                const uint8_t* cols = pa.rblob + lbq::kRefineHeader;
                for (int j0 = 0; j0 < pa.nsel; j0 += per) {
                    const int nb = min(per, pa.nsel - j0);
                    __syncthreads();   // the previous batch has been read
                    for (int jj = tid; jj < nb; jj += kThreads) {
                        const int c = pa.ridx[j0 + jj];
                        rsel_b[jj] = c >= 0 && c < pa.K ? c : -1;
                    }
                    __syncthreads();
                    for (int pi = tid; pi < nb * pieces; pi += kThreads) {
                        const int jj = pi / pieces, k = pi - jj * pieces;
                        const uint8_t* col = cols + static_cast<long long>(rsel_b[jj] >= 0 ? rsel_b[jj] : 0) * pa.rcb;
                        const uint8_t* src = k * 16 < ln        ? col + 16 * g0 + 16 * k
                                             : k * 16 < ln + ls ? col + rp.s_lo + (16 * k - ln)
                                                                : col + rp.z_lo + (16 * k - ln - ls);
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(raw + jj * lc + 16 * k)),
                                     "l"(src)
                                     : "memory");
                    }
                    // the x values load while the column copies are in flight
                    for (int jj = tid; jj < nb; jj += kThreads) {
                        const int c = rsel_b[jj];
                        if (c < 0) record_error(LBQ_ERR_VALUE);   // skipped: its x counts as 0
                        rx_b[jj] = c >= 0 ? __half2float(pa.x[c]) : 0.f;
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    __syncthreads();
                    accumulate(raw, rx_b, j0, nb);
                }
            }
            // each row of this problem: its word's partials, in slice order
            __syncthreads();
            for (int rl = rl0 + tid; rl < rl0 + static_cast<int>(n1 - n0); rl += kThreads) {
                const long long n = n0 + (rl - rl0);
                const int wi = (static_cast<int>(n >> 5) - g0) * 4 + static_cast<int>((n >> 2) & 3);
                const int e = static_cast<int>(n & 3) + (((n >> 4) & 1) ? 4 : 0);
                float tot = 0.f;
                for (int s2 = 0; s2 < WS; ++s2) tot += wpart[(s2 * nw + wi) * 8 + e];
                rfin[rl] = tot;
            }
        }
        __syncthreads();
    }
    if (check_rhdr) {
        const ProbArg& pa = a.p[blockIdx.x];
        const long long n_hdr = (static_cast<long long>(rhdr1.y) << 32) | rhdr1.x;
        const long long k_hdr = (static_cast<long long>(rhdr1.w) << 32) | rhdr1.z;
        if (rhdr0.x != 0x5251424Cu || rhdr0.y != 0x43345746u || rhdr0.z != lbq::kRefineVersion || n_hdr != pa.N ||
            k_hdr != pa.K)
            record_error(LBQ_ERR_FORMAT);
    }

    if (check_hdr) {
        const ProbArg& pa = a.p[blockIdx.x];
        const long long n_hdr = (static_cast<long long>(hdr1.y) << 32) | hdr1.x;
        const long long k_hdr = (static_cast<long long>(hdr1.w) << 32) | hdr1.z;
        if (hdr0.x != RC::kMagicLo || hdr0.y != RC::kMagicHi || hdr0.z != LBQ_FORMAT_VERSION_NUM || n_hdr != pa.N ||
            k_hdr != pa.K || static_cast<int>(hdr2.x) != pa.n_out)
            record_error(LBQ_ERR_FORMAT);
    }
    // combine: owned row blocks are already in yacc; shared ones add the parked
    // partials of their warps in warp order (deterministic)
    for (int i = tid; i < R * kTR * MB; i += kThreads) {
        const int m = i % MB, rr = i / MB;
        const int lu = rr / kTR, r = rr - lu * kTR;
        float y = yacc[i];
#pragma unroll 4
        for (int w = 0; w < NW; ++w) {
            if (seg[2 * w] == lu) y += part[((w * 2 + 0) * kTR + r) * MB + m];
            if (seg[2 * w + 1] == lu) y += part[((w * 2 + 1) * kTR + r) * MB + m];
        }
        const int u = u0 + lu;
        int q = qf;
        while (q + 1 < a.count && a.p[q + 1].ub <= u) ++q;
        const ProbArg& pa = a.p[q];
        const long long n = static_cast<long long>(u - pa.ub) * kTR + r;
        if (n < pa.N && m < mrows) {
            y *= 1.f / kUnit;
            if (refined && pa.nsel > 0)
                y += rfin[rr];
            if (a.y_f32)
                reinterpret_cast<float*>(pa.y)[m * pa.ldy + n] = y;
            else
                reinterpret_cast<__half*>(pa.y)[m * pa.ldy + n] = __float2half_rn(y);
        }
    }
}

// Self-test of the bounded wait every kernel uses: one thread waits on an
// mbarrier that nothing ever arrives on; after `limit_ns` the wait gives up, the
// error word records LBQ_ERR_TIMEOUT and the kernel returns normally.
__global__ void lbq_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait_bounded(&bar, 0, limit_ns)) record_error(LBQ_ERR_TIMEOUT);
    }
}

// ------------------------------------------------------------ host helpers

constexpr int kNumVariantsMax = 16;

struct DeviceInfo {
    bool init = false;
    bool ok = false;
    int sms = 0;
    int max_smem = 0;          // opt-in maximum per CTA
    unsigned* err_word = nullptr;   // device address of the error word
    bool attr_set[kNumVariantsMax] = {};
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

lbq_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LBQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LBQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return LBQ_ERR_CUDA;
        void* ew = nullptr;
        if (cudaGetSymbolAddress(&ew, g_lbq_error_word) != cudaSuccess) return LBQ_ERR_CUDA;
        d.err_word = static_cast<unsigned*>(ew);
        d.ok = (major == 10 && minor == 3);
        d.init = true;
    }
    if (!d.ok) return LBQ_ERR_UNSUPPORTED;
    *out = &d;
    return LBQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Kernel variants: (kind, MB activation planes, warps, records per item)
struct Variant {
    int kind, MB, NW, stage;
    const void* fn;
};
template <int KIND, int MB, int NW, int RPI>
Variant make_variant() {
    return Variant{KIND, MB, NW, Rec<KIND>::template stage<RPI>(),
                   reinterpret_cast<const void*>(&lbq_gemv_kernel<KIND, MB, NW, RPI>)};
}
constexpr int kNumVariants = 12;
static_assert(kNumVariants <= kNumVariantsMax, "DeviceInfo::attr_set holds one flag per variant");
constexpr int kVarW4 = 0, kVarW2 = 4, kVarW4Narrow = 5, kVarW2Narrow = 6, kVarW4One = 7, kVarW2One = 8;
// small-M variants (2, 4, 8 activation rows per pass) of each kind
constexpr int kVarW4Small[3] = {1, 2, 3}, kVarW2Small[3] = {9, 10, 11};
const Variant& variant(int v) {
    static const Variant table[kNumVariants] = {
        make_variant<kW4, 1, 16, 2>(),   // 0: 4-bit GEMV, two records per item
        make_variant<kW4, 2, 12, 1>(),   // 1..3: 4-bit small-M, 2 / 4 / 8 activation rows per pass
        make_variant<kW4, 4, 12, 1>(),
        make_variant<kW4, 8, 8, 1>(),
        make_variant<kW2, 1, 16, 2>(),   // 4: 2-bit codebook GEMV, two records per item
        make_variant<kW4, 1, 8, 1>(),    // 5, 6: fewer warps and one-record stages: room for very wide K;
                                         //       two CTAs fit an SM (small single calls, see run())
        make_variant<kW2, 1, 8, 1>(),
        make_variant<kW4, 1, 16, 1>(),   // 7, 8: one-record stages, for groups whose staging leaves no
        make_variant<kW2, 1, 16, 1>(),   //       room for two-record stages, and single 4-bit calls
        make_variant<kW2, 2, 12, 1>(),   // 9..11: 2-bit small-M, 2 / 4 / 8 activation rows per pass
        make_variant<kW2, 4, 12, 1>(),
        make_variant<kW2, 8, 8, 1>(),
    };
    return table[v];
}
// The variant to try when v does not fit a group's shared memory (-1: none):
// M = 1 goes from two-record stages to one-record stages to half the warps.
int fallback_variant(int v) {
    return v == kVarW4 ? kVarW4One : v == kVarW4One ? kVarW4Narrow : v == kVarW2 ? kVarW2One
                                                               : v == kVarW2One ? kVarW2Narrow : -1;
}

// One problem as the host entry points describe it.
struct HostProblem {
    const void* packed;
    int64_t N, K;
    int32_t n_out;
    const void* x;
    int64_t ldx;
    void* y;
    int64_t ldy;
    const void* refine = nullptr;   // selective refinement (M = 1)
    const int32_t* ridx = nullptr;
    int32_t nsel = 0;
};

// Fill the launch arguments of a group (without the partition).
lbq_status prepare_group(int kind, const HostProblem* P, int count, GroupArgs* a) {
    std::memset(a, 0, sizeof(*a));
    a->count = count;
    long long ub = 0;
    for (int i = 0; i < count; ++i) {
        lbq_layout L;
        lbq_status st = lbq_blob_layout(kind == kW4 ? LBQ_KIND_W4 : LBQ_KIND_W2CB, P[i].N, P[i].K, P[i].n_out, &L);
        if (st != LBQ_OK) return st;
        ProbArg& p = a->p[i];
        const uint8_t* b = static_cast<const uint8_t*>(P[i].packed);
        p.blob = b;
        p.area = b + L.area_offset;
        p.idx = reinterpret_cast<const int32_t*>(b + L.idx_offset);
        p.x = static_cast<const __half*>(P[i].x);
        p.y = P[i].y;
        p.ldx = P[i].ldx;
        p.ldy = P[i].ldy;
        p.N = P[i].N;
        p.K = P[i].K;
        p.rb_bytes = static_cast<long long>(L.row_block_bytes);
        p.recs = static_cast<int>(L.records);
        p.OT = static_cast<int>(L.outlier_records);
        p.out_last = p.OT > 0 ? static_cast<int>(L.row_block_bytes - L.records * L.record_bytes -
                                                 (L.outlier_records - 1) * L.outlier_record_bytes)
                              : 0;
        p.n_out = P[i].n_out;
        p.ub = static_cast<int>(ub);
        if (P[i].refine && P[i].nsel > 0) {
            p.rblob = static_cast<const uint8_t*>(P[i].refine);
            p.ridx = P[i].ridx;
            p.nsel = P[i].nsel;
            p.rcb = static_cast<long long>(lbq_refine_packed_bytes(P[i].N, 1)) - lbq::kRefineHeader;
        }
        ub += (P[i].N + kTR - 1) / kTR;
        if (ub > INT32_MAX / 2) return LBQ_ERR_SHAPE;
    }
    a->nunits = static_cast<int>(ub);
    // 2-bit codebook as FP16 byte tables for PRMT (otf-llm section 2, rounded once)
    const double cb[4] = {-1.52, -0.45, 0.45, 1.52};
    for (int c = 0; c < 4; ++c) {
        const uint16_t h = lbq::host_f64_to_f16(cb[c]);
        a->lut_lo |= uint32_t(h & 0xFF) << (8 * c);
        a->lut_hi |= uint32_t(h >> 8) << (8 * c);
    }
    return LBQ_OK;
}

int unit_end_host(const GroupArgs& a, int q) { return q + 1 < a.count ? a.p[q + 1].ub : a.nunits; }

// Persistent grid of <= one CTA per SM; CTA c owns a contiguous run of row
// blocks whose bytes are about 1/grid of the total.  Returns the largest
// staging area any CTA needs, and in *stg_ref_max the largest with the early
// refinement area added (M = 1); sets grid, cta_ub and rb_cap.
int partition(const DeviceInfo* dev, int MB, GroupArgs& a, int* grid, int* stg_ref_max) {
    long long total = 0;
    for (int q = 0; q < a.count; ++q) total += static_cast<long long>(unit_end_host(a, q) - a.p[q].ub) * a.p[q].rb_bytes;
    int G = dev->sms < kMaxGrid ? dev->sms : kMaxGrid;
    if (G > a.nunits) G = a.nunits;
    a.cta_ub[0] = 0;
    int q = 0;
    long long before = 0;   // bytes of the problems before q
    for (int c = 1; c < G; ++c) {
        const long long target = (total * c) / G;
        while (q + 1 < a.count && before + static_cast<long long>(unit_end_host(a, q) - a.p[q].ub) * a.p[q].rb_bytes <= target) {
            before += static_cast<long long>(unit_end_host(a, q) - a.p[q].ub) * a.p[q].rb_bytes;
            ++q;
        }
        // first row block of q whose start is at or past the target
        const long long into = target - before;
        long long u = a.p[q].ub + (into + a.p[q].rb_bytes - 1) / a.p[q].rb_bytes;
        if (u > unit_end_host(a, q)) u = unit_end_host(a, q);
        if (u < a.cta_ub[c - 1]) u = a.cta_ub[c - 1];
        a.cta_ub[c] = static_cast<int>(u);
    }
    a.cta_ub[G] = a.nunits;
    int rb_cap = 1, stg_max = 0;
    long long ref_max = 0;
    for (int c = 0; c < G; ++c) {
        const int u0 = a.cta_ub[c], u1 = a.cta_ub[c + 1];
        if (u1 - u0 > rb_cap) rb_cap = u1 - u0;
        int s = 0;
        long long r = 0;
        if (u1 > u0)
            for (int p = 0; p < a.count; ++p)
                if (a.p[p].ub < u1 && unit_end_host(a, p) > u0) {
                    s += staging_bytes(MB, a.p[p].recs, a.p[p].OT);
                    const int lo = u0 > a.p[p].ub ? u0 : a.p[p].ub;
                    const int hi = u1 < unit_end_host(a, p) ? u1 : unit_end_host(a, p);
                    const long long n0 = static_cast<long long>(lo - a.p[p].ub) * kTR;
                    long long n1 = static_cast<long long>(hi - a.p[p].ub) * kTR;
                    if (n1 > a.p[p].N) n1 = a.p[p].N;
                    if (MB == 1 && a.p[p].nsel > 0 && n1 > n0) r += ref_area_bytes(a.p[p].N, n0, n1, a.p[p].nsel);
                }
        if (s > stg_max) stg_max = s;
        if (s + r > ref_max) ref_max = s + r;
    }
    *stg_ref_max = ref_max > INT32_MAX / 2 ? INT32_MAX / 2 : static_cast<int>(ref_max);
    a.rb_cap = rb_cap;
    *grid = G;
    return stg_max;
}

// Stages per warp that fit next to the staging area; < 2 means "does not fit".
int stages_per_warp(const DeviceInfo* dev, const Variant& V, int rb_cap, int stg_max) {
    const FixedPlan f = fixed_plan(V.NW, V.stage, 0, V.MB, rb_cap);
    const int budget = dev->max_smem - f.total - stg_max - V.NW * kMaxStagesPerWarp * 8 - 128;
    const int spw = budget / (V.NW * V.stage);
    const int cap = V.MB == 1 ? kStagesM1 : kStagesMB;
    return spw > cap ? cap : spw;
}

// Plan one launch of variant vi over the group; LBQ_ERR_SHAPE when it does not fit.
lbq_status plan_group(const DeviceInfo* dev, int vi, GroupArgs& a, int* grid, size_t* smem) {
    const Variant& V = variant(vi);
    int stg_ref = 0;
    int stg_max = partition(dev, V.MB, a, grid, &stg_ref);
    // the early refinement area when it fits with the full ring, else the ring path
    a.rearly = 0;
    if (stg_ref > stg_max && stages_per_warp(dev, V, a.rb_cap, stg_ref) >= (V.MB == 1 ? kStagesM1 : kStagesMB)) {
        a.rearly = 1;
        stg_max = stg_ref;
    }
    const int spw = stages_per_warp(dev, V, a.rb_cap, stg_max);
    if (spw < 2) return LBQ_ERR_SHAPE;
    a.SPW = spw;
    *smem = static_cast<size_t>(fixed_plan(V.NW, V.stage, spw, V.MB, a.rb_cap).total + stg_max);
    return LBQ_OK;
}

lbq_status launch_planned(DeviceInfo* dev, int vi, const GroupArgs& a, int grid, size_t smem, void* stream,
                          uint32_t flags) {
    const Variant& V = variant(vi);
    if (!dev->attr_set[vi]) {
        if (cudaFuncSetAttribute(V.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev->max_smem) != cudaSuccess)
            return LBQ_ERR_CUDA;
        dev->attr_set[vi] = true;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(V.NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & LBQ_FLAG_PDL) ? 1 : 0;
    void* args[] = {const_cast<GroupArgs*>(&a)};
    if (cudaLaunchKernelExC(&cfg, V.fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    return LBQ_OK;
}

// One pass (mrows <= MB activation rows) over a group: the preferred variant,
// else (fallback) its fallback chain, else the group split in halves (launched back to
// back; the later half follows a kernel of this same call, which writes no blob,
// so it may overlap it).  With launches != nullptr nothing is launched and the
// kernels the pass would launch are counted instead.
lbq_status launch_pass(DeviceInfo* dev, int kind, int vi, bool fallback, const HostProblem* P, int count, int mrows,
                       bool y_f32, void* stream, uint32_t flags, int* launches) {
    static thread_local GroupArgs a;   // ~4 KB: kept off the caller's stack
    lbq_status st = prepare_group(kind, P, count, &a);
    if (st != LBQ_OK) return st;
    a.mrows = mrows;
    a.y_f32 = y_f32 ? 1 : 0;
    int grid = 0;
    size_t smem = 0;
    st = plan_group(dev, vi, a, &grid, &smem);
    for (int v = fallback ? fallback_variant(vi) : -1; st == LBQ_ERR_SHAPE && v >= 0; v = fallback_variant(v))
        st = plan_group(dev, v, a, &grid, &smem), vi = v;
    if (st == LBQ_OK) {
        if (launches) {
            ++*launches;
            return LBQ_OK;
        }
        return launch_planned(dev, vi, a, grid, smem, stream, flags);
    }
    if (st != LBQ_ERR_SHAPE || count == 1) return st;
    const int h = count / 2;
    st = launch_pass(dev, kind, vi, fallback, P, h, mrows, y_f32, stream, flags, launches);
    if (st != LBQ_OK) return st;
    return launch_pass(dev, kind, vi, fallback, P + h, count - h, mrows, y_f32, stream, flags | LBQ_FLAG_PDL,
                       launches);
}

lbq_status check_problem(const HostProblem& p, int M, lbq_dtype y_dtype) {
    if (!p.packed || !p.x || !p.y) return LBQ_ERR_NULL;
    if (p.N < 1 || p.N > INT32_MAX - 8 || p.K < 64 || p.K > lbq::kMaxK || p.K % 64 || p.n_out < 0 || p.n_out > p.K ||
        p.n_out > lbq::kMaxOutliers)
        return LBQ_ERR_SHAPE;
    if (p.ldx < p.K || p.ldy < p.N) return LBQ_ERR_SHAPE;
    if (M > 1 && static_cast<long long>(M) * p.ldx > (1ll << 40)) return LBQ_ERR_SHAPE;
    if (!aligned(p.packed, 16) || !aligned(p.x, 16) || p.ldx % 8 || !aligned(p.y, y_dtype == LBQ_F32 ? 4 : 2))
        return LBQ_ERR_ALIGN;
    return LBQ_OK;
}

// Passes of `MB`-row activation blocks over the group (offsets applied to x and y).
lbq_status run_passes(DeviceInfo* dev, int kind, int vi, bool fallback, int MB, const HostProblem* P, int count, int M,
                      bool f32, void* stream, uint32_t flags, int* launches) {
    const size_t ysz = f32 ? 4 : 2;
    HostProblem Q[kMaxGroup];
    for (int m0 = 0; m0 < M; m0 += MB) {
        for (int i = 0; i < count; ++i) {
            Q[i] = P[i];
            Q[i].x = static_cast<const __half*>(P[i].x) + m0 * P[i].ldx;
            Q[i].y = static_cast<uint8_t*>(P[i].y) + m0 * P[i].ldy * ysz;
        }
        // later passes follow a pass of this same call, which never writes a blob
        lbq_status st = launch_pass(dev, kind, vi, fallback, Q, count, M - m0 < MB ? M - m0 : MB, f32, stream,
                                    m0 == 0 ? flags : (flags | LBQ_FLAG_PDL), launches);
        if (st != LBQ_OK) return st;
    }
    return LBQ_OK;
}

// Every entry point ends here: validate, then one pass (M = 1), or passes of
// the narrowest small-M variant (2, 4 or 8 activation rows) covering M whose
// activation planes fit in shared memory for every problem on its own (a group
// is split into several launches when its problems do not fit together), or
// one GEMV pass per activation row when K is too wide for two planes.
lbq_status run(int kind, const HostProblem* P, int count, int M, lbq_dtype y_dtype, void* stream, uint32_t flags,
               int* launches) {
    if (count < 1 || count > kMaxGroup || M < 1 || M > lbq::kMaxM) return LBQ_ERR_SHAPE;
    if (y_dtype != LBQ_F16 && y_dtype != LBQ_F32) return LBQ_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i) {
        lbq_status st = check_problem(P[i], M, y_dtype);
        if (st != LBQ_OK) return st;
    }
    DeviceInfo* dev = nullptr;
    lbq_status st = device_info(&dev);
    if (st != LBQ_OK) return st;
    const bool f32 = y_dtype == LBQ_F32;
    const int vi = kind == kW4 ? kVarW4 : kVarW2;
    if (M == 1) {
        // one-record items for calls with fewer dense records than warps in the
        // grid (latency rather than bandwidth decides them) and for a single
        // large 4-bit problem, >= 4 records per warp (measured: 14336 x 4096
        // alone 9.1 us with one-record items, 9.8 us with two; grouped sweeps
        // are faster with two).  A single call with fewer than two records per
        // warp runs on the 8-warp variant, two of whose CTAs fit an SM: the next
        // launch's CTAs then start (and prefetch their weights) while this one
        // finishes, instead of after it (measured in chained calls: 1024 x 4096
        // 3.9 -> 2.9 us, 4096 x 4096 4.96 -> 4.79 us at 4-bit, 6.65 -> 5.98 us
        // at 2-bit; 14336 x 4096 is slower on 8 warps, 9.1 -> 9.6 us)
        long long recs = 0;
        for (int i = 0; i < count; ++i) recs += (P[i].N + kTR - 1) / kTR * ((P[i].K + 1023) / 1024);
        const long long warps = static_cast<long long>(dev->sms) * variant(vi).NW;
        const bool one = recs < warps || (kind == kW4 && count == 1 && recs >= 4 * warps);
        const bool dual = count == 1 && recs < 2 * warps;
        const int v0 = dual ? (kind == kW4 ? kVarW4Narrow : kVarW2Narrow) : one ? fallback_variant(vi) : vi;
        return launch_pass(dev, kind, v0, true, P, count, 1, f32, stream, flags, launches);
    }
    // M >= 16: the tensor-core kernels, one launch per problem
    if (M >= 16) {
        for (int i = 0; i < count; ++i) {
            const uint32_t fl = i == 0 ? flags : (flags | LBQ_FLAG_PDL);
            if (kind == kW2) {
                st = lbq::launch_w2_mma(P[i].packed, P[i].N, P[i].K, P[i].n_out, M, P[i].x, P[i].ldx, P[i].y,
                                        P[i].ldy, f32, dev->err_word, dev->max_smem, stream, fl, launches);
            } else if (launches) {
                ++*launches;
                st = LBQ_OK;
            } else {
                st = lbq::launch_w4_mma(P[i].packed, P[i].N, P[i].K, P[i].n_out, M, P[i].x, P[i].ldx, P[i].y,
                                        P[i].ldy, f32, dev->err_word, dev->sms, dev->max_smem, stream, fl);
            }
            if (st != LBQ_OK) return st;
        }
        return LBQ_OK;
    }
    const int* small = kind == kW4 ? kVarW4Small : kVarW2Small;
    int j = 0;
    while (j < 2 && variant(small[j]).MB < M) ++j;
    for (; j >= 0; --j) {
        bool fits = true;
        for (int i = 0; i < count && fits; ++i) {
            int n = 0;
            fits = launch_pass(dev, kind, small[j], false, P + i, 1, variant(small[j]).MB, f32, stream, 0u, &n) ==
                   LBQ_OK;
        }
        if (fits) break;
    }
    if (j >= 0)
        return run_passes(dev, kind, small[j], false, variant(small[j]).MB, P, count, M, f32, stream, flags,
                          launches);
    return run_passes(dev, kind, vi, true, 1, P, count, M, f32, stream, flags, launches);
}

lbq_status run_one(int kind, const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out, const void* x,
                   int64_t ldx, void* y, int64_t ldy, lbq_dtype y_dtype, void* stream, uint32_t flags) {
    if (!packed || !x || !y) return LBQ_ERR_NULL;
    HostProblem p{packed, N, K, n_out, x, ldx, y, ldy};
    return run(kind, &p, 1, M, y_dtype, stream, flags, nullptr);
}

lbq_status grouped(lbq_kind kind, const lbq_problem* problems, const lbq_refinement* refinements, int32_t count,
                   int32_t M, lbq_dtype y_dtype, void* stream, uint32_t flags, int* launches) {
    if (!problems) return LBQ_ERR_NULL;
    if (kind != LBQ_KIND_W4 && kind != LBQ_KIND_W2CB) return LBQ_ERR_UNSUPPORTED;
    if (count < 1 || count > kMaxGroup) return LBQ_ERR_SHAPE;
    HostProblem P[kMaxGroup];
    for (int i = 0; i < count; ++i) {
        const lbq_problem& q = problems[i];
        if (q.reserved != 0) return LBQ_ERR_SHAPE;
        P[i] = HostProblem{q.packed, q.N, q.K, q.n_out, q.x, q.ldx, q.y, q.ldy};
        if (refinements && refinements[i].refine) {
            const lbq_refinement& r = refinements[i];
            if (r.reserved != 0 || M != 1 || q.N % 64 || r.n_sel < 0 || r.n_sel > q.K) return LBQ_ERR_SHAPE;
            if (r.n_sel > 0 && !r.idx) return LBQ_ERR_NULL;
            if (!aligned(r.refine, 16) || (r.idx && !aligned(r.idx, 4))) return LBQ_ERR_ALIGN;
            P[i].refine = r.refine;
            P[i].ridx = r.idx;
            P[i].nsel = r.n_sel;
        }
    }
    return run(kind == LBQ_KIND_W4 ? kW4 : kW2, P, count, M, y_dtype, stream, flags, launches);
}

}  // namespace

namespace lbq {
lbq_status device_context(unsigned** err_word, int* sms) {
    DeviceInfo* dev = nullptr;
    const lbq_status st = device_info(&dev);
    if (st != LBQ_OK) return st;
    *err_word = dev->err_word;
    *sms = dev->sms;
    return LBQ_OK;
}
}  // namespace lbq

extern "C" {

lbq_status lbq_gemv_w4a16_ex(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16, void* y,
                             lbq_dtype y_dtype, void* stream, uint32_t flags) {
    return run_one(kW4, packed, 1, N, K, n_out, x_f16, K, y, N, y_dtype, stream, flags);
}

lbq_status lbq_gemv_w2cb_outlier_ex(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16,
                                    void* y, lbq_dtype y_dtype, void* stream, uint32_t flags) {
    return run_one(kW2, packed, 1, N, K, n_out, x_f16, K, y, N, y_dtype, stream, flags);
}

lbq_status lbq_gemv_w4a16(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16, void* y,
                          lbq_dtype y_dtype, void* stream) {
    return run_one(kW4, packed, 1, N, K, n_out, x_f16, K, y, N, y_dtype, stream, 0u);
}

lbq_status lbq_gemv_w2cb_outlier(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16,
                                 void* y, lbq_dtype y_dtype, void* stream) {
    return run_one(kW2, packed, 1, N, K, n_out, x_f16, K, y, N, y_dtype, stream, 0u);
}

lbq_status lbq_gemm_w4a16_smallM_ex(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                    const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                    void* stream, uint32_t flags) {
    return run_one(kW4, packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, flags);
}

lbq_status lbq_gemm_w4a16_smallM(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                 const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                 void* stream) {
    return run_one(kW4, packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, 0u);
}

lbq_status lbq_gemm_w2cb_outlier_smallM_ex(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                           const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                           void* stream, uint32_t flags) {
    return run_one(kW2, packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, flags);
}

lbq_status lbq_gemm_w2cb_outlier_smallM(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                        const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                        void* stream) {
    return run_one(kW2, packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, 0u);
}


lbq_status lbq_gemv_grouped(lbq_kind kind, const lbq_problem* problems, int32_t count, int32_t M,
                            lbq_dtype y_dtype, void* stream, uint32_t flags) {
    return grouped(kind, problems, nullptr, count, M, y_dtype, stream, flags, nullptr);
}

lbq_status lbq_gemv_grouped_refined(lbq_kind kind, const lbq_problem* problems, const lbq_refinement* refinements,
                                    int32_t count, lbq_dtype y_dtype, void* stream, uint32_t flags) {
    if (!refinements) return LBQ_ERR_NULL;
    return grouped(kind, problems, refinements, count, 1, y_dtype, stream, flags, nullptr);
}

lbq_status lbq_gemv_grouped_launches(lbq_kind kind, const lbq_problem* problems, int32_t count, int32_t M,
                                     lbq_dtype y_dtype, int32_t* launches) {
    if (!launches) return LBQ_ERR_NULL;
    int n = 0;
    const lbq_status st = grouped(kind, problems, nullptr, count, M, y_dtype, nullptr, 0u, &n);
    *launches = st == LBQ_OK ? n : 0;
    return st;
}

lbq_status lbq_selftest_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 5000000u) return LBQ_ERR_SHAPE;
    DeviceInfo* dev = nullptr;
    lbq_status st = device_info(&dev);
    if (st != LBQ_OK) return st;
    lbq_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_us) * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    return LBQ_OK;
}

lbq_status lbq_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_lbq_error_word, sizeof(word)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_lbq_error_word, &zero, sizeof(zero)) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    return static_cast<lbq_status>(word);
}

}  // extern "C"
