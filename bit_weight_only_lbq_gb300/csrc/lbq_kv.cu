// 4-bit Group-32 KV cache on sm_103a: quantise key / value states on write and
// read them back as FP16 (SPECTRA article, section 4.5 "Group-32 Microscaled
// 4-Bit Key-Value Cache and Dynamic Memory Tiering": states quantised into
// asymmetric 4-bit Group-32 blocks in place; the quantiser of section 3.4 /
// Appendix A, Proposition 2).
//
// A cached row (one token of one layer's K or V: heads x head_dim values) is one
// record: width/2 nibble bytes (byte k of a group = q_k | q_{k+16} << 4), width/32
// FP16 scales, width/64 zero-point bytes (z_{2m} | z_{2m+1} << 4), padded to 16
// bytes.  Appending a decode step writes one record per tensor.
//
// GB300 design: the write is tiny and latency-bound (one token = a few hundred
// bytes), the read is memory-bound (0.58 B read, 2 B written per value).
//  * quantise: one warp (and CTA) per pair of groups (64 values: both share a
//    zero-point byte), a half warp per group, two values per lane (the two
//    nibbles of one record byte); min / max by shuffles; the statistics and
//    the divisions are FP64 with IEEE rounding and round-half-to-even, exactly
//    the host recipe, so the records are bit-identical to the host / reference
//    quantiser;
//  * dequantise: a thread turns one group (one 16-byte nibble load, its scale
//    and zero point) into 32 FP16 values ((q - z) s16 is exact in FP32, then
//    one rounding) written with four 16-byte stores.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kThreads = 256;

// One warp per pair of groups (the two share a zero-point byte), one CTA per
// warp (the FP64 work of a token's few warps spreads over as many SMs): lanes
// 0..15 take group 2p, lanes 16..31 group 2p + 1, lane l of a half the values
// l and l + 16 of its group - exactly the two nibbles of record byte l.  Min /
// max of the FP16 values are exact in FP32 (half-warp shuffles); the scale, the
// zero point and the codes follow in FP64 with IEEE rounding.
constexpr int kQThreads = 32;

__global__ void __launch_bounds__(kQThreads) lbq_kv_quantize_kernel(const __half* __restrict__ x, long long ldx,
                                                                    int rows, int width, uint8_t* __restrict__ cache,
                                                                    long long first_row, long long rec_bytes) {
    const int pairs = width / 64;
    const int lane = threadIdx.x & 31;
    const long long item = (static_cast<long long>(blockIdx.x) * kQThreads + threadIdx.x) >> 5;
    if (item >= static_cast<long long>(rows) * pairs) return;   // warp-uniform
    const int row = static_cast<int>(item / pairs), p = static_cast<int>(item % pairs);
    const int l = lane & 15;
    const __half* xg = x + row * ldx + p * 64 + (lane >> 4) * 32;
    const float va = __half2float(xg[l]), vb = __half2float(xg[l + 16]);
    float mn = fminf(va, vb), mx = fmaxf(va, vb);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const double wmin = static_cast<double>(mn), wmax = static_cast<double>(mx);
    // s = max((wmax - wmin) / 15, 1e-8), z = clamp(round(-wmin / s)), q = clamp(round(w / s + z))
    const double s = fmax(__ddiv_rn(__dsub_rn(wmax, wmin), 15.0), 1e-8);
    const double z = fmin(fmax(rint(__ddiv_rn(-wmin, s)), 0.0), 15.0);
    const uint32_t qa =
        static_cast<uint32_t>(fmin(fmax(rint(__dadd_rn(__ddiv_rn(static_cast<double>(va), s), z)), 0.0), 15.0));
    const uint32_t qb =
        static_cast<uint32_t>(fmin(fmax(rint(__dadd_rn(__ddiv_rn(static_cast<double>(vb), s), z)), 0.0), 15.0));
    uint8_t* rec = cache + (first_row + row) * rec_bytes;
    rec[p * 32 + lane] = static_cast<uint8_t>(qa | (qb << 4));
    const uint32_t s16 = __half_as_ushort(__double2half(s)), zi = static_cast<uint32_t>(z);
    const uint32_t s16_hi = __shfl_down_sync(0xffffffffu, s16, 16), z_hi = __shfl_down_sync(0xffffffffu, zi, 16);
    if (lane == 0) {
        // scales of groups 2p, 2p + 1 (4-byte aligned: width / 2 is a multiple of 32), their zero byte
        *reinterpret_cast<uint32_t*>(rec + width / 2 + p * 4) = s16 | (s16_hi << 16);
        rec[width / 2 + width / 16 + p] = static_cast<uint8_t>(zi | (z_hi << 4));
    }
    if (p == 0 && lane == 0)   // the record's padding reads as zero
        for (long long b = width / 2 + width / 16 + width / 64; b < rec_bytes; ++b) rec[b] = 0;
}

// A thread per group: one 16-byte load of its nibbles, its scale and zero
// point, four 16-byte stores of its 32 FP16 values.
__global__ void __launch_bounds__(kThreads) lbq_kv_dequant_kernel(const uint8_t* __restrict__ cache,
                                                                  long long first_row, int rows, int width,
                                                                  long long rec_bytes, __half* __restrict__ out,
                                                                  long long ldo) {
    const int per_row = width / 32;                      // groups per row
    const long long item = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    if (item >= static_cast<long long>(rows) * per_row) return;
    const int row = static_cast<int>(item / per_row), g = static_cast<int>(item % per_row);
    const uint8_t* rec = cache + (first_row + row) * rec_bytes;
    const uint4 qq = *reinterpret_cast<const uint4*>(rec + g * 16);
    const float s = __half2float(*reinterpret_cast<const __half*>(rec + width / 2 + g * 2));
    const uint32_t zb = rec[width / 2 + width / 16 + (g >> 1)];
    const float z = static_cast<float>((g & 1) ? (zb >> 4) : (zb & 15u));
    const uint32_t w[4] = {qq.x, qq.y, qq.z, qq.w};
    uint4* o = reinterpret_cast<uint4*>(out + row * ldo + g * 32);
#pragma unroll
    for (int h = 0; h < 2; ++h) {            // low nibbles: k = 0..15, high nibbles: k = 16..31
#pragma unroll
        for (int c = 0; c < 2; ++c) {        // 8 values per 16-byte store
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t word = w[2 * c + (j >> 1)];
                const uint32_t b0 = (word >> (16 * (j & 1))) & 0xFFu, b1 = (word >> (16 * (j & 1) + 8)) & 0xFFu;
                // (q - z) s: exact in FP32 (5-bit integer times FP16), one rounding to FP16
                const float v0 = (static_cast<float>((b0 >> (4 * h)) & 15u) - z) * s;
                const float v1 = (static_cast<float>((b1 >> (4 * h)) & 15u) - z) * s;
                const __half2 h2 = __floats2half2_rn(v0, v1);
                p[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            o[2 * h + c] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool shape_ok(int64_t width) { return width >= 64 && width <= lbq::kMaxK && width % 64 == 0; }

}  // namespace

extern "C" {

size_t lbq_kv_record_bytes(int64_t width) {
    if (!shape_ok(width)) return 0;
    return static_cast<size_t>((width / 2 + width / 16 + width / 64 + 15) / 16 * 16);
}

lbq_status lbq_kv_quantize(const void* x_f16, int64_t ldx, int64_t rows, int64_t width, void* cache,
                           int64_t first_row, void* stream) {
    if (rows == 0) return LBQ_OK;
    if (!x_f16 || !cache) return LBQ_ERR_NULL;
    if (!shape_ok(width) || rows < 0 || rows > INT32_MAX || first_row < 0 || ldx < width) return LBQ_ERR_SHAPE;
    if (!aligned(x_f16, 16) || ldx % 8 || !aligned(cache, 16)) return LBQ_ERR_ALIGN;
    unsigned* err = nullptr;
    int sms = 0;
    const lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    const long long warps = rows * (width / 64);
    if (warps > 0x7FFFFFFFll) return LBQ_ERR_SHAPE;   // one CTA per warp
    lbq_kv_quantize_kernel<<<static_cast<unsigned>(warps), kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __half*>(x_f16), ldx, static_cast<int>(rows), static_cast<int>(width),
        static_cast<uint8_t*>(cache), first_row, static_cast<long long>(lbq_kv_record_bytes(width)));
    if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    return LBQ_OK;
}

lbq_status lbq_kv_dequant(const void* cache, int64_t first_row, int64_t rows, int64_t width, void* out_f16,
                          int64_t ldo, void* stream) {
    if (rows == 0) return LBQ_OK;
    if (!cache || !out_f16) return LBQ_ERR_NULL;
    if (!shape_ok(width) || rows < 0 || rows > INT32_MAX || first_row < 0 || ldo < width) return LBQ_ERR_SHAPE;
    if (!aligned(cache, 16) || !aligned(out_f16, 16) || ldo % 8) return LBQ_ERR_ALIGN;
    unsigned* err = nullptr;
    int sms = 0;
    const lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    const long long items = rows * (width / 32);
    lbq_kv_dequant_kernel<<<static_cast<unsigned>((items + kThreads - 1) / kThreads), kThreads, 0,
                            static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(cache), first_row, static_cast<int>(rows), static_cast<int>(width),
        static_cast<long long>(lbq_kv_record_bytes(width)), static_cast<__half*>(out_f16), ldo);
    if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    return LBQ_OK;
}

}  // extern "C"
