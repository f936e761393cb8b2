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
//  * the blob stores each (4-row block x 32-group block) as one contiguous
//    record (packed codes, then scales/S, then zeros/Z), so a tile of GPL
//    records is one contiguous range of HBM;
//  * one persistent CTA per SM; each warp owns a private ring of shared-memory
//    stages that its lane 0 refills with one bulk copy per tile
//    (cp.async.bulk, the Tensor Memory Accelerator's 1-D mode) completing on
//    an mbarrier, so each SM keeps tens of KB in flight with no per-thread
//    address arithmetic;
//  * a tile is 4 output rows x (32 * GPL) groups; a lane owns GPL groups and
//    keeps their activations in registers for the tile's 4 rows; the CTA's
//    tiles are cut into contiguous per-warp ranges (split-K inside the CTA
//    when it owns few row blocks), partial rows are combined in warp order;
//  * 4-bit: a nibble masked in place is an exact FP16 subnormal (q * 2^-24);
//    a mixed-precision FMA (FP16 inputs, exact FP32 product) accumulates
//    q * x in FP32, and the zero point enters once per group as z * sum(x);
//  * 2-bit: a byte-permute (PRMT) table lookup turns 2-bit codes into FP16
//    codebook values; S multiplies the codebook dot product, Z the group's
//    activation sum;
//  * outlier columns are streamed as extra 4 x 256 FP16 tiles of the same row
//    block and accumulated before the cross-lane reduction;
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

constexpr int kTR = 4;                 // output rows per tile (row block)
constexpr int kOutCols = 256;          // outlier columns per outlier tile
constexpr int kOutTileBytes = kTR * kOutCols * 2;     // 2048
constexpr int kMaxStagesPerWarp = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum Kind { kW4 = 0, kW2 = 1 };

constexpr int round128(int b) { return (b + 127) / 128 * 128; }

// Dense record (one row block x 32 groups, the blob's unit) and tile geometry:
// a tile is GPL consecutive records of one row block; a lane owns one group of
// each record.
template <int KIND, int GPL>
struct Geo {
    static constexpr int kPacked = KIND == kW4 ? 16 : 8;               // packed bytes per (row, group)
    static constexpr int kOff1 = kTR * 32 * kPacked;                   // scales / S
    static constexpr int kOff2 = kOff1 + kTR * 32 * 2;                 // zeros / Z
    static constexpr int kRec = kOff2 + (KIND == kW4 ? kTR * 16 : kTR * 32 * 2);   // 2368 / 1536
    static constexpr int kDense = GPL * kRec;
    static constexpr int kStage = round128(kDense > kOutTileBytes ? kDense : kOutTileBytes);
    static constexpr uint32_t kMagicLo = 0x5751424Cu;                            // "LBQW"
    static constexpr uint32_t kMagicHi = KIND == kW4 ? 0x32334734u : 0x32334332u;  // "4G32" / "2C32"
};

struct GemvArgs {
    const uint8_t* blob;
    const uint8_t* area;   // first row block
    const __half* x;       // activation rows, leading dimension ldx (elements)
    const int32_t* idx;
    void* y;               // output rows, leading dimension ldy (elements)
    long long N, K;
    long long ldx, ldy;
    long long rb_bytes;    // bytes per row block
    int recs;              // dense records per row block
    int mrows;             // activation rows in this launch (<= MB of the kernel)
    int n_out;
    int y_f32;
    int n_rb;              // row blocks of kTR rows
    int KT;                // dense tiles per row block (records / GPL, rounded up)
    int OT;                // outlier records per row block
    int SPW;               // stages per warp
    int rb_cap;            // most row blocks any CTA owns
    uint32_t lut_lo, lut_hi;   // 2-bit codebook: low / high bytes of the FP16 centroids
};

// ----------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
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

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_bounded(bar, parity, kWaitLimitNs);
}

// One contiguous global -> shared bulk copy (bytes % 16 == 0, both ends 16-byte
// aligned) completing on an mbarrier, with an L2 eviction-priority hint.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
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
// half index of element k (0..K) of one activation plane
template <int KIND>
__device__ __forceinline__ int x_half_index(int k) {
    const int g = k >> 5, kk = k & 31;
    int slot;
    if (KIND == kW4) {
        const int hi = kk >> 4, r = kk & 15;
        slot = 8 * (r >> 2) + 2 * ((r & 1) + 2 * hi) + ((r >> 1) & 1);
    } else {
        const int v = kk >> 4, r = kk & 15;
        slot = 16 * v + 4 * (r & 3) + 2 * (r >> 3) + ((r >> 2) & 1);
    }
    return x_chunk_index(g, slot >> 3) * 8 + (slot & 7);
}

// --------------------------------------------------------------- tile math

// 4-bit dense tile.  A nibble masked in place is the FP16 subnormal q * 2^-24
// (low nibble) or 16 q * 2^-24 (high nibble); the mixed-precision FMA turns it
// into the exact FP32 product with x.  Per group: dot = lo + hi / 16 =
// 2^-24 sum_k q_k x_k and w.x = s (sum_k q_k x_k - z X_g) = 2^24 s (dot - z X_g 2^-24);
// the final 2^24 is applied once per output.
template <int MB, int GPL>
__device__ __forceinline__ void w4_dense_tile(const uint8_t* st, int nrec, const uint4* xq, int xq_plane,
                                              const float* xs24, int xs_plane, int mrows, int lane,
                                              float (&acc)[MB][kTR]) {
    using G = Geo<kW4, GPL>;
#pragma unroll
    for (int h = 0; h < GPL; ++h) {
        if (h >= nrec) break;                          // short last tile
        const uint8_t* rec = st + h * G::kRec;
        const uint4* qw = reinterpret_cast<const uint4*>(rec);
        const __half* sc = reinterpret_cast<const __half*>(rec + G::kOff1);
        const uint8_t* zp = rec + G::kOff2;
        const int gl = lane;                           // group within the record
        if constexpr (MB == 1) {
            const uint4 xr[4] = {xq[h * 128], xq[h * 128 + 32], xq[h * 128 + 64], xq[h * 128 + 96]};
            const float xsz = xs24[h * 32];
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                const uint4 q = qw[r * 32 + gl];
                const float s = __half2float(sc[r * 32 + gl]);
                const uint32_t zb = zp[r * 16 + (gl >> 1)];
                const float zf = static_cast<float>((zb >> ((lane & 1) * 4)) & 15u);
                float l0 = 0.f, l1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w = u4w(q, j), w8 = w >> 8;
                    l0 = fma2_mixed(w & 0x000F000Fu, xr[j].x, l0);
                    l1 = fma2_mixed(w8 & 0x000F000Fu, xr[j].y, l1);
                    h0 = fma2_mixed(w & 0x00F000F0u, xr[j].z, h0);
                    h1 = fma2_mixed(w8 & 0x00F000F0u, xr[j].w, h1);
                }
                const float t = fmaf(-zf, xsz, fmaf(h0 + h1, 0.0625f, l0 + l1));
                acc[0][r] = fmaf(s, t, acc[0][r]);
            }
        } else {
            uint32_t u[kTR][16];
            float s[kTR], zf[kTR];
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                const uint4 q = qw[r * 32 + gl];
                s[r] = __half2float(sc[r * 32 + gl]);
                const uint32_t zb = zp[r * 16 + (gl >> 1)];
                zf[r] = static_cast<float>((zb >> ((lane & 1) * 4)) & 15u);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w = u4w(q, j), w8 = w >> 8;
                    u[r][4 * j + 0] = w & 0x000F000Fu;
                    u[r][4 * j + 1] = w8 & 0x000F000Fu;
                    u[r][4 * j + 2] = w & 0x00F000F0u;
                    u[r][4 * j + 3] = w8 & 0x00F000F0u;
                }
            }
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                if (m < mrows) {
                    const uint4* xp = xq + m * xq_plane + h * 128;
                    const uint4 xr[4] = {xp[0], xp[32], xp[64], xp[96]};
                    const float xsz = xs24[m * xs_plane + h * 32];
#pragma unroll
                    for (int r = 0; r < kTR; ++r) {
                        float l0 = 0.f, l1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            l0 = fma2_mixed(u[r][4 * j + 0], xr[j].x, l0);
                            l1 = fma2_mixed(u[r][4 * j + 1], xr[j].y, l1);
                            h0 = fma2_mixed(u[r][4 * j + 2], xr[j].z, h0);
                            h1 = fma2_mixed(u[r][4 * j + 3], xr[j].w, h1);
                        }
                        const float t = fmaf(-zf[r], xsz, fmaf(h0 + h1, 0.0625f, l0 + l1));
                        acc[m][r] = fmaf(s[r], t, acc[m][r]);
                    }
                }
            }
        }
    }
}

// 2-bit dense tile: four codes -> PRMT selector (c, c+4 per code) -> two FP16
// codebook pairs; w.x = S sum_k C[q_k] x_k + Z X_g.
template <int GPL>
__device__ __forceinline__ void w2_dense_tile(const uint8_t* st, int nrec, const uint4* xq, const float* xsum,
                                              int lane, uint32_t lut_lo, uint32_t lut_hi, float (&acc)[kTR]) {
    using G = Geo<kW2, GPL>;
#pragma unroll
    for (int h = 0; h < GPL; ++h) {
        if (h >= nrec) break;                          // short last tile
        const uint8_t* rec = st + h * G::kRec;
        const uint2* cw = reinterpret_cast<const uint2*>(rec);
        const __half* Sg = reinterpret_cast<const __half*>(rec + G::kOff1);
        const __half* Zg = reinterpret_cast<const __half*>(rec + G::kOff2);
        const int gl = lane;
        const uint4 xr[4] = {xq[h * 128], xq[h * 128 + 32], xq[h * 128 + 64], xq[h * 128 + 96]};
        const float xs = xsum[h * 32];
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
            const uint2 c = cw[r * 32 + gl];
            const float S = __half2float(Sg[r * 32 + gl]);
            const float Z = __half2float(Zg[r * 32 + gl]);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const uint32_t w = v ? c.y : c.x;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint32_t t = (w >> (2 * s)) & 0x03030303u;
                    const uint32_t sel = t * 0x11u + 0x40404040u;     // nibbles (c, c + 4) per code
                    const uint32_t h01 = prmt(lut_lo, lut_hi, sel);
                    const uint32_t h23 = prmt(lut_lo, lut_hi, sel >> 16);
                    const int mw = (v * 4 + s) * 2;                    // word of the group's 64 x bytes
                    d[s & 1] = fma2_mixed(h01, u4w(xr[mw >> 2], mw & 3), d[s & 1]);
                    d[2 + (s & 1)] = fma2_mixed(h23, u4w(xr[(mw + 1) >> 2], (mw + 1) & 3), d[2 + (s & 1)]);
                }
            }
            acc[r] = fmaf(S, (d[0] + d[1]) + (d[2] + d[3]), fmaf(Z, xs, acc[r]));
        }
    }
}

// One outlier tile: lane owns outlier columns [ot*256 + lane*8, +8) of the 4
// rows; xo_tile + m * xo_plane holds x[idx] of activation row m.  `scale`
// converts to the unit of the dense accumulator (2^-24 for 4-bit, 1 for 2-bit).
template <int MB>
__device__ __forceinline__ void outlier_tile(const uint8_t* st, const __half* xo_tile, int xo_plane, int mrows,
                                             int lane, float scale, float (&acc)[MB][kTR]) {
    uint4 v[kTR];
#pragma unroll
    for (int r = 0; r < kTR; ++r) v[r] = reinterpret_cast<const uint4*>(st)[r * 32 + lane];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        if (m < mrows) {
            const uint4 xv = reinterpret_cast<const uint4*>(xo_tile + m * xo_plane)[lane];
#pragma unroll
            for (int r = 0; r < kTR; ++r) {
                float a0 = fma2_mixed(v[r].x, xv.x, 0.f);
                float a1 = fma2_mixed(v[r].y, xv.y, 0.f);
                a0 = fma2_mixed(v[r].z, xv.z, a0);
                a1 = fma2_mixed(v[r].w, xv.w, a1);
                acc[m][r] = fmaf(a0 + a1, scale, acc[m][r]);
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

struct SmemPlan {
    int ring, xs, xsum, xo, omask, yacc, part, seg, bars, total;
};

// NW warps, rb_cap: most row blocks a CTA owns; MB: activation planes.
__host__ __device__ inline SmemPlan smem_plan(int NW, int stage, int KTg, int OT, int SPW, int MB, int rb_cap) {
    // KTg: 32-group blocks covered by the dense tiles (KT * GPL)
    SmemPlan p;
    int off = 0;
    p.ring = off;
    off += NW * SPW * stage;
    p.xs = off;
    off += MB * KTg * 32 * 64;
    p.xsum = off;
    off += MB * KTg * 32 * 4;
    p.xo = off;
    off += MB * OT * kOutCols * 2;
    p.omask = off;
    off += KTg * 32 * 4;                   // one bit per k: outlier channel
    p.yacc = off;
    off += rb_cap * kTR * MB * 4;
    p.part = off;
    off += NW * 2 * kTR * MB * 4;
    p.seg = off;
    off += NW * 2 * 4;                     // per warp: first and last row block it touched
    off = (off + 7) / 8 * 8;
    p.bars = off;
    off += NW * SPW * 8;
    p.total = off + 128;   // slack for aligning the base to 128 bytes
    return p;
}

template <int KIND, int MB, int NW, int GPL>
__global__ void __launch_bounds__(NW * 32, 1) lbq_gemv_kernel(const __grid_constant__ GemvArgs a) {
    using G = Geo<KIND, GPL>;
    constexpr int kThreads = NW * 32;
    constexpr float kUnit = KIND == kW4 ? 5.9604644775390625e-8f : 1.f;   // 2^-24 for the 4-bit products
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // align by offsetting the shared array itself, so the compiler keeps the
    // shared address space (LDS with immediate offsets, no generic addressing)
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int KTg = a.KT * GPL;
    const SmemPlan P = smem_plan(NW, G::kStage, KTg, a.OT, a.SPW, MB, a.rb_cap);
    uint8_t* ring = smem + P.ring;
    uint4* xs = reinterpret_cast<uint4*>(smem + P.xs);
    float* xsum = reinterpret_cast<float*>(smem + P.xsum);
    __half* xo = reinterpret_cast<__half*>(smem + P.xo);
    uint32_t* omask = reinterpret_cast<uint32_t*>(smem + P.omask);
    float* yacc = reinterpret_cast<float*>(smem + P.yacc);
    float* part = reinterpret_cast<float*>(smem + P.part);
    int* seg = reinterpret_cast<int*>(smem + P.seg);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int SPW = a.SPW;
    const int TPR = a.KT + a.OT;                    // tiles per row block
    const int ngroups = KTg * 32;                   // groups per (padded) activation plane
    const int xq_plane = ngroups * 4;               // uint4 chunks per plane
    const int xo_plane = a.OT * kOutCols;
    const int mrows = a.mrows;
    const int rb_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * a.n_rb) / gridDim.x);
    const int rb_end = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * a.n_rb) / gridDim.x);
    const int R = rb_end - rb_begin;
    const int n_tiles = R * TPR;                    // this CTA's tiles, row block major
    // each warp takes a contiguous share of the CTA's tiles (split-K when row blocks are few)
    const int w_begin = (warp * n_tiles) / NW;
    const int w_end = ((warp + 1) * n_tiles) / NW;
    const int my_tiles = w_end - w_begin;
    uint64_t* my_bars = bars + warp * SPW;
    uint8_t* my_ring = ring + warp * SPW * G::kStage;
    const uint64_t policy = policy_evict_first();

    // issue pointer (lane 0 only): next tile's row block and k tile
    int i_rb = w_begin / TPR, i_kk = w_begin - (w_begin / TPR) * TPR, i_slot = 0;
    auto issue_next = [&]() {
        uint8_t* dst = my_ring + i_slot * G::kStage;
        uint64_t* bar = my_bars + i_slot;
        const uint8_t* rb_src = a.area + static_cast<long long>(rb_begin + i_rb) * a.rb_bytes;
        if (i_kk < a.KT) {
            const int r0 = i_kk * GPL;
            const int nrec = a.recs - r0 < GPL ? a.recs - r0 : GPL;
            const uint32_t bytes = static_cast<uint32_t>(nrec * G::kRec);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(dst, rb_src + static_cast<long long>(r0) * G::kRec, bytes, bar, policy);
        } else {
            mbar_arrive_expect_tx(bar, kOutTileBytes);
            bulk_load(dst, rb_src + static_cast<long long>(a.recs) * G::kRec +
                               static_cast<long long>(i_kk - a.KT) * kOutTileBytes,
                      kOutTileBytes, bar, policy);
        }
        if (++i_kk == TPR) {
            i_kk = 0;
            ++i_rb;
        }
        if (++i_slot == SPW) i_slot = 0;
    };

    // barriers, then start the weight stream before waiting on the previous grid
    if (lane == 0) {
        for (int s = 0; s < SPW; ++s) mbar_init(my_bars + s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const int pre = my_tiles < SPW ? my_tiles : SPW;
        for (int t = 0; t < pre; ++t) issue_next();
    }
    // blob header: loaded now (three 16-byte loads in flight), compared after the main loop,
    // so the check never delays this CTA's prologue
    uint4 hdr0 = make_uint4(0u, 0u, 0u, 0u), hdr1 = hdr0, hdr2 = hdr0;
    if (blockIdx.x == 0 && tid == 0) {
        const uint4* h = reinterpret_cast<const uint4*>(a.blob);
        hdr0 = h[0];
        hdr1 = h[1];
        hdr2 = h[2];
    }
    // outlier-channel bitmask and the row accumulators (no dependence on the previous grid)
    for (int i = tid; i < ngroups; i += kThreads) omask[i] = 0u;
    for (int i = tid; i < R * kTR * MB; i += kThreads) yacc[i] = 0.f;
    pdl_trigger();
    if (a.n_out > 0) {
        __syncthreads();
        for (int j = tid; j < a.n_out; j += kThreads) {
            const int k = a.idx[j];
            if (k >= 0 && k < a.K)
                atomicOr(&omask[k >> 5], 1u << (k & 31));
            else
                record_error(LBQ_ERR_OUTLIER_IDX);   // corrupted blob: never index outside x
        }
    }
    __syncthreads();
    pdl_wait();

    // stage x: a thread takes whole groups (four 16-byte loads), zeroes outlier
    // channels, writes the permuted chunks and the group sum X~_g (times kUnit)
    for (int base = tid; base < MB * ngroups; base += kThreads * 2) {
        uint4 raw[2][4];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int i = base + b * kThreads;
            const int m = i / ngroups, g = i - m * ngroups;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                raw[b][j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < MB * ngroups && m < mrows && g * 32 < a.K)
                    raw[b][j] = *reinterpret_cast<const uint4*>(a.x + m * a.ldx + g * 32 + j * 8);
            }
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int i = base + b * kThreads;
            if (i < MB * ngroups) {
                const int m = i / ngroups, g = i - m * ngroups;
                uint32_t n[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    n[4 * j + 0] = raw[b][j].x;
                    n[4 * j + 1] = raw[b][j].y;
                    n[4 * j + 2] = raw[b][j].z;
                    n[4 * j + 3] = raw[b][j].w;
                }
                const uint32_t om = a.n_out > 0 ? omask[g] : 0u;
                if (om) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t keep = ((om >> (2 * e)) & 1u ? 0xFFFF0000u : 0xFFFFFFFFu) &
                                              ((om >> (2 * e + 1)) & 1u ? 0x0000FFFFu : 0xFFFFFFFFu);
                        n[e] &= keep;
                    }
                }
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    s0 = fma2_mixed(n[e], 0x3C003C00u, s0);         // + x_{2e} + x_{2e+1}
                    s1 = fma2_mixed(n[e + 1], 0x3C003C00u, s1);
                }
                xsum[i] = (s0 + s1) * kUnit;
                uint4* dst = xs + m * xq_plane;
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[x_chunk_index(g, j)] = permuted_chunk<KIND>(n, j);
            }
        }
    }
    // x[idx] of every activation row, from global memory (the unmasked values)
    for (int i = tid; i < MB * xo_plane; i += kThreads) {
        const int m = i / xo_plane, j = i - m * xo_plane;
        __half v = __float2half(0.f);
        if (j < a.n_out && m < mrows) {
            const int k = a.idx[j];
            if (k >= 0 && k < a.K) v = a.x[m * a.ldx + k];
        }
        xo[i] = v;
    }
    __syncthreads();

    // main loop: this warp's tiles through its ring; a segment is a run of tiles of one row block
    bool ok = true;
    int c_rb = w_begin / TPR, c_kk = w_begin - (w_begin / TPR) * TPR, c_slot = 0;
    uint32_t c_phase = 0;
    const int first_rb = my_tiles > 0 ? c_rb : -1, last_rb = my_tiles > 0 ? (w_end - 1) / TPR : -1;
    if (lane == 0) {
        seg[2 * warp] = first_rb;
        seg[2 * warp + 1] = last_rb != first_rb ? last_rb : -1;
    }
    float acc[MB][kTR];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int r = 0; r < kTR; ++r) acc[m][r] = 0.f;
    int t = 0;
    for (; t < my_tiles; ++t) {
        const bool got = mbar_wait(my_bars + c_slot, c_phase);
        if (!__all_sync(0xffffffffu, got)) {   // warp-uniform: any lane timing out aborts the warp
            ok = false;
            break;
        }
        const uint8_t* st = my_ring + c_slot * G::kStage;
        if (c_kk < a.KT) {
            const uint4* xq = xs + c_kk * GPL * 128 + lane;
            const float* xsg = xsum + c_kk * GPL * 32 + lane;
            const int nrec = a.recs - c_kk * GPL;            // records in this tile (>= GPL except at the end)
            if constexpr (KIND == kW4)
                w4_dense_tile<MB, GPL>(st, nrec, xq, xq_plane, xsg, ngroups, mrows, lane, acc);
            else
                w2_dense_tile<GPL>(st, nrec, xq, xsg, lane, a.lut_lo, a.lut_hi, acc[0]);
        } else {
            outlier_tile<MB>(st, xo + (c_kk - a.KT) * kOutCols, xo_plane, mrows, lane, kUnit, acc);
        }
        __syncwarp();
        // refill the stage: every lane's reads of it completed before __syncwarp
        if (lane == 0 && t + SPW < my_tiles) issue_next();
        if (++c_slot == SPW) {
            c_slot = 0;
            c_phase ^= 1u;
        }
        // end of a segment: reduce over lanes and park the row partials
        if (++c_kk == TPR || t + 1 == my_tiles) {
            const int pslot = (c_rb == first_rb) ? 0 : (c_rb == last_rb ? 1 : -1);
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                if (m < mrows) {
                    const float tot = reduce_rows4(acc[m], lane);
                    if ((lane & 7) == 0) {
                        const int r = lane >> 3;
                        if (pslot < 0)
                            yacc[(c_rb * kTR + r) * MB + m] = tot;             // row block owned by this warp alone
                        else
                            part[((warp * 2 + pslot) * kTR + r) * MB + m] = tot;
                    }
                }
#pragma unroll
                for (int r = 0; r < kTR; ++r) acc[m][r] = 0.f;
            }
            if (c_kk == TPR) {
                c_kk = 0;
                ++c_rb;
            }
        }
    }
    if (!ok) {
        if (lane == 0) {
            record_error(LBQ_ERR_TIMEOUT);
            // drain the copies this warp still has in flight before its shared memory goes away
            const int outstanding = (my_tiles - t) < SPW ? (my_tiles - t) : SPW;
            for (int u = 0; u < outstanding; ++u) {
                const int slot = (c_slot + u) % SPW;
                const uint32_t ph = (slot >= c_slot) ? c_phase : (c_phase ^ 1u);
                mbar_wait_bounded(my_bars + slot, ph, kWaitLimitNs / 8);
            }
        }
        __syncwarp();
    }
    __syncthreads();

    if (blockIdx.x == 0 && tid == 0) {
        const long long n_hdr = (static_cast<long long>(hdr1.y) << 32) | hdr1.x;
        const long long k_hdr = (static_cast<long long>(hdr1.w) << 32) | hdr1.z;
        if (hdr0.x != G::kMagicLo || hdr0.y != G::kMagicHi || hdr0.z != LBQ_FORMAT_VERSION_NUM || n_hdr != a.N ||
            k_hdr != a.K || static_cast<int>(hdr2.x) != a.n_out)
            record_error(LBQ_ERR_FORMAT);
    }
    // combine: owned row blocks are already in yacc; shared ones add the parked
    // partials of their warps in warp order (deterministic)
    for (int i = tid; i < R * kTR * MB; i += kThreads) {
        const int m = i % MB, rr = i / MB;
        const int rbl = rr / kTR, r = rr - rbl * kTR;
        float y = yacc[i];
#pragma unroll 4
        for (int w = 0; w < NW; ++w) {
            if (seg[2 * w] == rbl) y += part[((w * 2 + 0) * kTR + r) * MB + m];
            if (seg[2 * w + 1] == rbl) y += part[((w * 2 + 1) * kTR + r) * MB + m];
        }
        const long long n = static_cast<long long>(rb_begin + rbl) * kTR + r;
        if (n < a.N && m < mrows) {
            y *= 1.f / kUnit;
            if (a.y_f32)
                reinterpret_cast<float*>(a.y)[m * a.ldy + n] = y;
            else
                reinterpret_cast<__half*>(a.y)[m * a.ldy + n] = __float2half_rn(y);
        }
    }
}

// ------------------------------------------------------------ host helpers

constexpr int kNumVariantsMax = 8;

struct DeviceInfo {
    bool init = false;
    bool ok = false;
    int sms = 0;
    int max_smem = 0;          // opt-in maximum per CTA
    int smem_per_sm = 0;
    int smem_reserved = 0;     // per CTA, reserved by the system
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
            cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return LBQ_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        d.init = true;
    }
    if (!d.ok) return LBQ_ERR_UNSUPPORTED;
    *out = &d;
    return LBQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Kernel variants: (kind, MB activation planes, warps, groups per lane)
struct Variant {
    int kind, MB, NW, GPL, stage;
    const void* fn;
};
template <int KIND, int MB, int NW, int GPL>
Variant make_variant() {
    return Variant{KIND, MB, NW, GPL, Geo<KIND, GPL>::kStage,
                   reinterpret_cast<const void*>(&lbq_gemv_kernel<KIND, MB, NW, GPL>)};
}
constexpr int kNumVariants = 7;
const Variant& variant(int v) {
    static const Variant table[kNumVariants] = {
        make_variant<kW4, 1, 16, 2>(),   // 0: 4-bit GEMV
        make_variant<kW4, 2, 8, 1>(),    // 1..3: 4-bit small-M, 2 / 4 / 8 activation rows per pass
        make_variant<kW4, 4, 8, 1>(),
        make_variant<kW4, 8, 8, 1>(),
        make_variant<kW2, 1, 16, 2>(),   // 4: 2-bit codebook GEMV
        make_variant<kW4, 1, 8, 1>(),    // 5, 6: smaller-footprint GEMVs for very wide K
        make_variant<kW2, 1, 8, 1>(),
    };
    return table[v];
}

lbq_status prepare_args(const Variant& V, const void* packed, int64_t N, int64_t K, int32_t n_out, GemvArgs* a) {
    lbq_layout L;
    lbq_status st = lbq_blob_layout(V.kind == kW4 ? LBQ_KIND_W4 : LBQ_KIND_W2CB, N, K, n_out, &L);
    if (st != LBQ_OK) return st;
    std::memset(a, 0, sizeof(*a));
    const uint8_t* b = static_cast<const uint8_t*>(packed);
    a->blob = b;
    a->area = b + L.area_offset;
    a->idx = reinterpret_cast<const int32_t*>(b + L.idx_offset);
    a->rb_bytes = static_cast<long long>(L.row_block_bytes);
    a->recs = static_cast<int>(L.records);
    a->N = N;
    a->K = K;
    a->n_out = n_out;
    a->n_rb = static_cast<int>((N + kTR - 1) / kTR);
    a->KT = (a->recs + V.GPL - 1) / V.GPL;
    a->OT = static_cast<int>(L.outlier_records);
    // 2-bit codebook as FP16 byte tables for PRMT (otf-llm section 2, rounded once)
    const double cb[4] = {-1.52, -0.45, 0.45, 1.52};
    for (int c = 0; c < 4; ++c) {
        const uint16_t h = lbq::host_f64_to_f16(cb[c]);
        a->lut_lo |= uint32_t(h & 0xFF) << (8 * c);
        a->lut_hi |= uint32_t(h >> 8) << (8 * c);
    }
    return LBQ_OK;
}

// Stages per warp that fit in `budget` bytes next to the activation planes;
// < 2 means "does not fit".
int stages_per_warp(const Variant& V, int budget, int KT, int OT, int rb_cap) {
    const SmemPlan fixed = smem_plan(V.NW, V.stage, KT * V.GPL, OT, 0, V.MB, rb_cap);
    int spw = (budget - fixed.total - V.NW * kMaxStagesPerWarp * 8) / (V.NW * V.stage);
    return spw > kMaxStagesPerWarp ? kMaxStagesPerWarp : spw;
}

struct LaunchShape {
    int grid, rb_cap, SPW;
};

// One persistent CTA per SM (fewer when there are fewer row blocks), each
// owning a contiguous, balanced run of row blocks.
LaunchShape launch_shape(const DeviceInfo* dev, const Variant& V, int n_rb, int KT, int OT) {
    LaunchShape L;
    L.grid = n_rb < dev->sms ? n_rb : dev->sms;
    L.rb_cap = (n_rb + L.grid - 1) / L.grid;
    L.SPW = stages_per_warp(V, dev->max_smem, KT, OT, L.rb_cap);
    return L;
}

lbq_status launch_variant(DeviceInfo* dev, int vi, GemvArgs& a, void* stream, uint32_t flags) {
    const Variant& V = variant(vi);
    const LaunchShape S = launch_shape(dev, V, a.n_rb, a.KT, a.OT);
    if (S.SPW < 2) return LBQ_ERR_SHAPE;
    a.rb_cap = S.rb_cap;
    a.SPW = S.SPW;
    const SmemPlan P = smem_plan(V.NW, V.stage, a.KT * V.GPL, a.OT, a.SPW, V.MB, a.rb_cap);
    if (!dev->attr_set[vi]) {
        if (cudaFuncSetAttribute(V.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev->max_smem) != cudaSuccess)
            return LBQ_ERR_CUDA;
        dev->attr_set[vi] = true;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(S.grid));
    cfg.blockDim = dim3(V.NW * 32);
    cfg.dynamicSmemBytes = P.total;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & LBQ_FLAG_PDL) ? 1 : 0;
    void* args[] = {&a};
    if (cudaLaunchKernelExC(&cfg, V.fn, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    return LBQ_OK;
}

lbq_status check_common(const void* packed, int64_t N, int64_t K, int32_t n_out, lbq_dtype y_dtype) {
    if (N < 1 || N > INT32_MAX - 8 || K < 64 || K > lbq::kMaxK || K % 64 || n_out < 0 || n_out > K ||
        n_out > lbq::kMaxOutliers)
        return LBQ_ERR_SHAPE;
    if (y_dtype != LBQ_F16 && y_dtype != LBQ_F32) return LBQ_ERR_UNSUPPORTED;
    if (!aligned(packed, 16)) return LBQ_ERR_ALIGN;
    return LBQ_OK;
}

// Launch a GEMV-shaped call (mrows activation rows, one pass) on the preferred
// variant, or on its smaller-footprint fallback when shared memory is short.
lbq_status launch_one(DeviceInfo* dev, int vi, int vfallback, const void* packed, int64_t N, int64_t K,
                      int32_t n_out, const void* x, int64_t ldx, void* y, int64_t ldy, int mrows, lbq_dtype y_dtype,
                      void* stream, uint32_t flags) {
    GemvArgs a;
    lbq_status st = prepare_args(variant(vi), packed, N, K, n_out, &a);
    if (st != LBQ_OK) return st;
    if (vfallback >= 0 && launch_shape(dev, variant(vi), a.n_rb, a.KT, a.OT).SPW < 2) {
        vi = vfallback;
        st = prepare_args(variant(vi), packed, N, K, n_out, &a);
        if (st != LBQ_OK) return st;
    }
    a.x = static_cast<const __half*>(x);
    a.y = y;
    a.ldx = ldx;
    a.ldy = ldy;
    a.mrows = mrows;
    a.y_f32 = (y_dtype == LBQ_F32);
    return launch_variant(dev, vi, a, stream, flags);
}

lbq_status launch_gemv(int kind, const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x, void* y,
                       lbq_dtype y_dtype, void* stream, uint32_t flags) {
    if (!packed || !x || !y) return LBQ_ERR_NULL;
    lbq_status st = check_common(packed, N, K, n_out, y_dtype);
    if (st != LBQ_OK) return st;
    if (!aligned(x, 16) || !aligned(y, y_dtype == LBQ_F32 ? 4 : 2)) return LBQ_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != LBQ_OK) return st;
    return kind == kW4 ? launch_one(dev, 0, 5, packed, N, K, n_out, x, K, y, N, 1, y_dtype, stream, flags)
                       : launch_one(dev, 4, 6, packed, N, K, n_out, x, K, y, N, 1, y_dtype, stream, flags);
}

lbq_status launch_smallm(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out, const void* X,
                         int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype, void* stream, uint32_t flags) {
    if (!packed || !X || !Y) return LBQ_ERR_NULL;
    lbq_status st = check_common(packed, N, K, n_out, y_dtype);
    if (st != LBQ_OK) return st;
    if (M < 1 || M > lbq::kMaxM || ldx < K || ldy < N) return LBQ_ERR_SHAPE;
    if (!aligned(X, 16) || ldx % 8 || !aligned(Y, y_dtype == LBQ_F32 ? 4 : 2)) return LBQ_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != LBQ_OK) return st;
    if (M == 1) return launch_one(dev, 0, 5, packed, N, K, n_out, X, ldx, Y, ldy, 1, y_dtype, stream, flags);
    // widest activation block that fits in shared memory next to the weight ring,
    // then the narrowest one that still covers M in a single pass
    GemvArgs a;
    st = prepare_args(variant(1), packed, N, K, n_out, &a);     // variants 1..3 share the tiling
    if (st != LBQ_OK) return st;
    const size_t ysz = y_dtype == LBQ_F32 ? 4 : 2;
    if (launch_shape(dev, variant(1), a.n_rb, a.KT, a.OT).SPW < 2) {
        // K too wide for two activation planes: one GEMV pass per row
        for (int m = 0; m < M; ++m) {
            st = launch_one(dev, 0, 5, packed, N, K, n_out, static_cast<const __half*>(X) + m * ldx, ldx,
                            static_cast<uint8_t*>(Y) + m * ldy * ysz, ldy, 1, y_dtype, stream,
                            m == 0 ? flags : LBQ_FLAG_PDL);
            if (st != LBQ_OK) return st;
        }
        return LBQ_OK;
    }
    int vmax = 3;
    while (vmax > 1 && launch_shape(dev, variant(vmax), a.n_rb, a.KT, a.OT).SPW < 4) --vmax;
    int vi = 1;
    while (vi < vmax && variant(vi).MB < M) ++vi;
    const int MB = variant(vi).MB;
    a.ldx = ldx;
    a.ldy = ldy;
    a.y_f32 = (y_dtype == LBQ_F32);
    for (int m0 = 0; m0 < M; m0 += MB) {
        a.x = static_cast<const __half*>(X) + m0 * ldx;
        a.y = static_cast<uint8_t*>(Y) + m0 * ldy * ysz;
        a.mrows = M - m0 < MB ? M - m0 : MB;
        // later passes follow a pass of this same call, which never writes the blob
        st = launch_variant(dev, vi, a, stream, m0 == 0 ? flags : LBQ_FLAG_PDL);
        if (st != LBQ_OK) return st;
    }
    return LBQ_OK;
}

}  // namespace

extern "C" {

lbq_status lbq_gemv_w4a16_ex(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16, void* y,
                             lbq_dtype y_dtype, void* stream, uint32_t flags) {
    return launch_gemv(kW4, packed, N, K, n_out, x_f16, y, y_dtype, stream, flags);
}

lbq_status lbq_gemv_w2cb_outlier_ex(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16,
                                    void* y, lbq_dtype y_dtype, void* stream, uint32_t flags) {
    return launch_gemv(kW2, packed, N, K, n_out, x_f16, y, y_dtype, stream, flags);
}

lbq_status lbq_gemv_w4a16(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16, void* y,
                          lbq_dtype y_dtype, void* stream) {
    return launch_gemv(kW4, packed, N, K, n_out, x_f16, y, y_dtype, stream, 0u);
}

lbq_status lbq_gemv_w2cb_outlier(const void* packed, int64_t N, int64_t K, int32_t n_out, const void* x_f16,
                                 void* y, lbq_dtype y_dtype, void* stream) {
    return launch_gemv(kW2, packed, N, K, n_out, x_f16, y, y_dtype, stream, 0u);
}

lbq_status lbq_gemm_w4a16_smallM_ex(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                    const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                    void* stream, uint32_t flags) {
    return launch_smallm(packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, flags);
}

lbq_status lbq_gemm_w4a16_smallM(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                 const void* X_f16, int64_t ldx, void* Y, int64_t ldy, lbq_dtype y_dtype,
                                 void* stream) {
    return launch_smallm(packed, M, N, K, n_out, X_f16, ldx, Y, ldy, y_dtype, stream, 0u);
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
