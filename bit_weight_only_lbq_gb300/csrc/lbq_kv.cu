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
//  * quantise: one warp per pair of groups (64 values: both share a zero-point
//    byte), a lane per value of each group; min / max by warp shuffles; the
//    statistics and the division are FP64 with IEEE rounding and
//    round-half-to-even, exactly the host recipe, so the records are
//    bit-identical to the host / reference quantiser;
//  * dequantise: a thread turns one 8-byte nibble load into 8 FP16 values
//    ((q - z) s16 is exact in FP32, then one rounding) and writes them with one
//    16-byte store.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ double warp_min(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmin(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_max(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One warp per pair of groups (the two share a zero-point byte): lane l holds
// value l of each group; min / max by shuffles, then each lane quantises its two
// values, lanes 0..15 write the nibble bytes, lane 0 the scales and the zero byte.
__global__ void __launch_bounds__(kThreads) lbq_kv_quantize_kernel(const __half* __restrict__ x, long long ldx,
                                                                   int rows, int width, uint8_t* __restrict__ cache,
                                                                   long long first_row, long long rec_bytes) {
    const int pairs = width / 64;
    const int lane = threadIdx.x & 31;
    const long long item = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    if (item >= static_cast<long long>(rows) * pairs) return;   // warp-uniform
    const int row = static_cast<int>(item / pairs), p = static_cast<int>(item % pairs);
    const __half* xr = x + row * ldx + p * 64;
    uint8_t* rec = cache + (first_row + row) * rec_bytes;
    uint32_t zpair = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int g = 2 * p + h;
        const double w = static_cast<double>(__half2float(xr[h * 32 + lane]));
        const double wmin = warp_min(w), wmax = warp_max(w);
        // s = max((wmax - wmin) / 15, 1e-8), z = clamp(round(-wmin / s)), q = clamp(round(w / s + z))
        const double s = fmax(__ddiv_rn(__dsub_rn(wmax, wmin), 15.0), 1e-8);
        const double z = fmin(fmax(rint(__ddiv_rn(-wmin, s)), 0.0), 15.0);
        const uint32_t q = static_cast<uint32_t>(fmin(fmax(rint(__dadd_rn(__ddiv_rn(w, s), z)), 0.0), 15.0));
        const uint32_t q_hi = __shfl_down_sync(0xffffffffu, q, 16);          // value lane + 16
        if (lane < 16) rec[g * 16 + lane] = static_cast<uint8_t>(q | (q_hi << 4));
        if (lane == 0) *reinterpret_cast<__half*>(rec + width / 2 + g * 2) = __double2half(s);
        zpair |= static_cast<uint32_t>(z) << (4 * h);
    }
    if (lane == 0) rec[width / 2 + width / 16 + p] = static_cast<uint8_t>(zpair);
    if (p == 0 && lane == 0)   // the record's padding reads as zero
        for (long long b = width / 2 + width / 16 + width / 64; b < rec_bytes; ++b) rec[b] = 0;
}

__global__ void __launch_bounds__(kThreads) lbq_kv_dequant_kernel(const uint8_t* __restrict__ cache,
                                                                  long long first_row, int rows, int width,
                                                                  long long rec_bytes, __half* __restrict__ out,
                                                                  long long ldo) {
    const int per_row = width / 8;                       // 8 values per thread
    const long long item = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    if (item >= static_cast<long long>(rows) * per_row) return;
    const int row = static_cast<int>(item / per_row), c0 = static_cast<int>(item % per_row) * 8;
    const uint8_t* rec = cache + (first_row + row) * rec_bytes;
    const int g = c0 >> 5, k0 = c0 & 31;
    const uint2 qq = *reinterpret_cast<const uint2*>(rec + g * 16 + (k0 & 15));
    const float s = __half2float(*reinterpret_cast<const __half*>(rec + width / 2 + g * 2));
    const uint32_t zb = rec[width / 2 + width / 16 + (g >> 1)];
    const int z = static_cast<int>((g & 1) ? (zb >> 4) : (zb & 15u));
    const int sh = k0 >= 16 ? 4 : 0;
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b0 = ((j < 2 ? qq.x : qq.y) >> (16 * (j & 1))) & 0xFFu;
        const uint32_t b1 = ((j < 2 ? qq.x : qq.y) >> (16 * (j & 1) + 8)) & 0xFFu;
        const float v0 = static_cast<float>(static_cast<int>((b0 >> sh) & 15u) - z) * s;
        const float v1 = static_cast<float>(static_cast<int>((b1 >> sh) & 15u) - z) * s;
        const __half2 h2 = __floats2half2_rn(v0, v1);
        p[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(out + row * ldo + c0) = make_uint4(p[0], p[1], p[2], p[3]);
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
    const long long per_cta = kThreads / 32;
    lbq_kv_quantize_kernel<<<static_cast<unsigned>((warps + per_cta - 1) / per_cta), kThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
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
    const long long items = rows * (width / 8);
    lbq_kv_dequant_kernel<<<static_cast<unsigned>((items + kThreads - 1) / kThreads), kThreads, 0,
                            static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(cache), first_row, static_cast<int>(rows), static_cast<int>(width),
        static_cast<long long>(lbq_kv_record_bytes(width)), static_cast<__half*>(out_f16), ldo);
    if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    return LBQ_OK;
}

}  // extern "C"
