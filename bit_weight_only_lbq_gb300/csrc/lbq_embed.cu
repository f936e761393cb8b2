// Fused embedding row gather on sm_103a: dequantise only the rows of the
// requested token ids from a packed table (SPECTRA article, section 4.3
// "SpectraFusedEmbedding: Dynamic Row-Gather Dequantization"; the table is a
// blob of either kind, rows = vocabulary entries, K = hidden size).
//
// An output row is the row of the matrix the blob applies: the dense part
// dequantised (4-bit (q - z) s, exact in FP32; 2-bit S C[q] + Z, in FP64) and
// rounded once to the output type, then the exact FP16 outlier columns.
//
// GB300 design: the gather is a pure copy-and-widen of a few KB per token
// (0.58 B read and 2 B written per element at 4-bit), so it is a plain
// memory-bound kernel: a CTA of 256 threads covers two 1,024-column records of
// one token's row, a thread dequantises 8 consecutive columns from one 8-byte
// (4-bit) or 2-byte (2-bit) load and writes them with one 16-byte (FP16) or
// two 16-byte (FP32) stores; a second small kernel writes the outlier columns
// of each row after the dense pass (stream order, no overlap of writers).

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

struct EmbedArgs {
    const uint8_t* blob;
    const int32_t* ids;
    void* out;
    unsigned* err;
    long long area_off, rb_bytes, rec_bytes, idx_off;
    int V, D, recs, n_out, T, out_f16, kind;
    unsigned short cb[4];   // 2-bit codebook, FP16 bits
};

constexpr int kThreads = 256;

__device__ __forceinline__ bool row_of(const EmbedArgs& a, int t, int* n) {
    const int v = a.ids[t];
    if (v < 0 || v >= a.V) {
        if (threadIdx.x == 0) atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_VALUE));
        return false;
    }
    *n = v;
    return true;
}

__global__ void __launch_bounds__(kThreads) lbq_embed_dense_kernel(const __grid_constant__ EmbedArgs a) {
    const int t = blockIdx.x, tid = threadIdx.x;
    if (t == 0 && blockIdx.y == 0 && tid == 0) {
        const uint32_t* h = reinterpret_cast<const uint32_t*>(a.blob);
        long long n_hdr, k_hdr;
        memcpy(&n_hdr, a.blob + 16, 8);
        memcpy(&k_hdr, a.blob + 24, 8);
        const uint32_t magic1 = a.kind == LBQ_KIND_W4 ? 0x32334734u : 0x32334332u;   // "4G32" / "2C32"
        if (h[0] != 0x5751424Cu || h[1] != magic1 || h[2] != LBQ_FORMAT_VERSION_NUM || n_hdr != a.V || k_hdr != a.D)
            atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_FORMAT));
    }
    int n;
    if (!row_of(a, t, &n)) return;
    const int rec = 2 * blockIdx.y + (tid >> 7), w = tid & 127;
    const int c0 = rec * 1024 + 8 * w;                      // first of this thread's 8 columns
    if (rec >= a.recs || c0 >= a.D) return;
    const int g = w >> 2, k0 = 8 * (w & 3);                 // group in the record, first k in the group
    const int r = n & 3;
    const uint8_t* rp = a.blob + a.area_off + static_cast<long long>(n >> 2) * a.rb_bytes +
                        static_cast<long long>(rec) * a.rec_bytes;
    float v32[8];
    if (a.kind == LBQ_KIND_W4) {
        // byte k of a group = q_k | q_{k+16} << 4: columns k0..k0+7 are the low
        // (k0 < 16) or high nibbles of bytes k0 % 16 .. + 7
        const uint2 qq = *reinterpret_cast<const uint2*>(rp + r * 512 + g * 16 + (k0 & 15));
        const float s = __half2float(*reinterpret_cast<const __half*>(rp + 2048 + r * 64 + g * 2));
        const uint32_t zb = rp[2304 + r * 16 + (g >> 1)];
        const int z = static_cast<int>((g & 1) ? (zb >> 4) : (zb & 15u));
        const int sh = k0 >= 16 ? 4 : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = ((j < 4 ? qq.x : qq.y) >> (8 * (j & 3))) & 0xFFu;
            const int q = static_cast<int>((byte >> sh) & 15u);
            v32[j] = static_cast<float>(q - z) * s;         // exact: 5-bit integer times FP16
        }
        if (a.out_f16) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h2 = __floats2half2_rn(v32[2 * j], v32[2 * j + 1]);
                p[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + static_cast<long long>(t) * a.D + c0) =
                make_uint4(p[0], p[1], p[2], p[3]);
        } else {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<long long>(t) * a.D + c0);
            o[0] = make_float4(v32[0], v32[1], v32[2], v32[3]);
            o[1] = make_float4(v32[4], v32[5], v32[6], v32[7]);
        }
    } else {
        // 2-bit: byte = q0 | q1 << 2 | q2 << 4 | q3 << 6 for four consecutive k;
        // S C[q] + Z in FP64, rounded once to the output type
        const uint32_t codes = *reinterpret_cast<const unsigned short*>(rp + r * 256 + g * 8 + k0 / 4);
        const double S = static_cast<double>(__half2float(*reinterpret_cast<const __half*>(rp + 1024 + r * 64 + g * 2)));
        const double Z = static_cast<double>(__half2float(*reinterpret_cast<const __half*>(rp + 1280 + r * 64 + g * 2)));
        double v64[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = static_cast<int>((codes >> (2 * j)) & 3u);
            const double c = static_cast<double>(__half2float(__ushort_as_half(a.cb[q])));
            v64[j] = __dadd_rn(__dmul_rn(S, c), Z);          // no contraction: product, then sum
        }
        if (a.out_f16) {
            __half hv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) hv[j] = __double2half(v64[j]);
            *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + static_cast<long long>(t) * a.D + c0) =
                *reinterpret_cast<const uint4*>(hv);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v32[j] = __double2float_rn(v64[j]);
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<long long>(t) * a.D + c0);
            o[0] = make_float4(v32[0], v32[1], v32[2], v32[3]);
            o[1] = make_float4(v32[4], v32[5], v32[6], v32[7]);
        }
    }
}

// The outlier columns of each gathered row: exact FP16 values from the row
// block's outlier records (256 columns each, the last one trimmed).
__global__ void __launch_bounds__(kThreads) lbq_embed_outlier_kernel(const __grid_constant__ EmbedArgs a) {
    const int t = blockIdx.x;
    int n;
    if (!row_of(a, t, &n)) return;
    const int r = n & 3;
    const uint8_t* ob = a.blob + a.area_off + static_cast<long long>(n >> 2) * a.rb_bytes +
                        static_cast<long long>(a.recs) * a.rec_bytes;
    const int32_t* idx = reinterpret_cast<const int32_t*>(a.blob + a.idx_off);
    const int padded = (a.n_out + lbq::kOutlierColAlign - 1) / lbq::kOutlierColAlign * lbq::kOutlierColAlign;
    for (int j = threadIdx.x; j < a.n_out; j += kThreads) {
        const int orec = j / lbq::kOutlierCols;
        const int width = min(lbq::kOutlierCols, padded - orec * lbq::kOutlierCols);
        const __half v = *reinterpret_cast<const __half*>(ob + orec * (4 * lbq::kOutlierCols * 2) +
                                                          (r * width + j % lbq::kOutlierCols) * 2);
        const int col = idx[j];
        if (col < 0 || col >= a.D) {
            atomicCAS(a.err, 0u, static_cast<unsigned>(LBQ_ERR_FORMAT));
            continue;
        }
        if (a.out_f16)
            static_cast<__half*>(a.out)[static_cast<long long>(t) * a.D + col] = v;
        else
            static_cast<float*>(a.out)[static_cast<long long>(t) * a.D + col] = __half2float(v);
    }
}

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

}  // namespace

extern "C" {

lbq_status lbq_embed_gather(lbq_kind kind, const void* packed, int64_t V, int64_t D, int32_t n_out,
                            const int32_t* ids, int32_t T, void* out, lbq_dtype out_dtype, void* stream) {
    if (!packed || (T > 0 && (!ids || !out))) return LBQ_ERR_NULL;
    if (kind != LBQ_KIND_W4 && kind != LBQ_KIND_W2CB) return LBQ_ERR_UNSUPPORTED;
    if (out_dtype != LBQ_F16 && out_dtype != LBQ_F32) return LBQ_ERR_UNSUPPORTED;
    if (V < 1 || V > INT32_MAX || D < 64 || D > lbq::kMaxK || D % 64 || n_out < 0 || n_out > D || T < 0)
        return LBQ_ERR_SHAPE;
    if (T == 0) return LBQ_OK;
    if (!aligned(packed, 16) || !aligned(ids, 4) || !aligned(out, 16)) return LBQ_ERR_ALIGN;
    lbq_layout L;
    lbq_status st = lbq_blob_layout(kind, V, D, n_out, &L);
    if (st != LBQ_OK) return st;
    unsigned* err = nullptr;
    int sms = 0;
    st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    EmbedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.blob = static_cast<const uint8_t*>(packed);
    a.ids = ids;
    a.out = out;
    a.err = err;
    a.area_off = static_cast<long long>(L.area_offset);
    a.rb_bytes = static_cast<long long>(L.row_block_bytes);
    a.rec_bytes = static_cast<long long>(L.record_bytes);
    a.idx_off = static_cast<long long>(L.idx_offset);
    a.V = static_cast<int>(V);
    a.D = static_cast<int>(D);
    a.recs = static_cast<int>(L.records);
    a.n_out = n_out;
    a.T = T;
    a.out_f16 = out_dtype == LBQ_F16 ? 1 : 0;
    a.kind = kind;
    const double cbk[4] = {-1.52, -0.45, 0.45, 1.52};   // otf-llm section 2 codebook (FP16-rounded)
    for (int c = 0; c < 4; ++c) a.cb[c] = lbq::host_f64_to_f16(cbk[c]);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    lbq_embed_dense_kernel<<<dim3(static_cast<unsigned>(T), static_cast<unsigned>((a.recs + 1) / 2)), kThreads, 0,
                             s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    if (n_out > 0) {
        lbq_embed_outlier_kernel<<<static_cast<unsigned>(T), kThreads, 0, s>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LBQ_ERR_CUDA;
    }
    return LBQ_OK;
}

}  // extern "C"
