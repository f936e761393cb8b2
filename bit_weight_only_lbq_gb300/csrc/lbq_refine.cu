// Selective weight refinement on sm_103a: exact per-chunk top-k channel
// selection and the gathered 4-bit column correction
//     y' = y + sum_{i in S(x)} x_i C[:, i]
// (StrataFlux paper, section 3 "Weight Refinement", Eq. 2, and "Channel
// selection": k channels of largest |x_i| per chunk of 1,024 input channels;
// Appendix "StrataFlux Implementation": exact radix-sort selection instead of
// bucket selection).  C is stored as one contiguous record per input channel
// (lbq_pack_refine), so a selected column is fetched in one piece.
//
// GB300 design:
//  * selection: one CTA of 1,024 threads per chunk, one channel per thread.
//    The key (|x| as its 15 FP16 magnitude bits, then 1023 - channel) is unique,
//    so a most-significant-digit radix select (9 + 8 + 8 bits, one
//    shared-memory histogram per pass, a warp-parallel scan of the bins with
//    16-byte loads) finds
//    the k-th largest key exactly; ties in |x| go to the lower channel.  The
//    selected channels are written in ascending order with a ballot prefix sum.
//  * apply: one CTA per 256 output rows, W warps (8, or 32 for selections of
//    more than 128 columns) taking every W-th selected column, the indices of
//    a warp's next 32 columns loaded at once; a lane owns one 32-bit nibble
//    word (8 rows) of a group and accumulates x_i (q - z) s in FP32 ((q - z) s
//    is exact in FP32); the W warps' partial rows are added in warp order
//    (deterministic) and added to y.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kChunk = lbq::kRefineChunk;
static_assert(kChunk == 1024, "the selection runs one thread per channel of a 1,024-channel chunk");

// Index scratch of lbq_refine_noalloc: one array per device, shared by every
// call.  64 chunks (K <= 65536) x 256 channels (k <= 256) = 16384 indices, 64 KB.
constexpr int kNoAllocIdxMax = (lbq::kMaxK / lbq::kRefineChunk) * lbq::kRefineMaxK;
static_assert(kNoAllocIdxMax >= ((lbq::kMaxK + lbq::kRefineChunk - 1) / lbq::kRefineChunk) * lbq::kRefineMaxK,
              "the scratch holds the selection of every valid (K, k)");
__device__ __align__(256) int32_t g_refine_idx_scratch[kNoAllocIdxMax];
constexpr int kApplyRows = 256;
constexpr int kApplyWarpsMax = 32;
constexpr int kApplyWideFrom = 128;   // selections longer than this use 32 warps

// Warp-parallel search of the histogram from its top bin down: the bin in which
// the running count reaches `remaining`; returns it and the count above it.  A
// lane reads its 8 or 16 consecutive bins with 16-byte loads (a 2-way bank
// conflict instead of 16-way for one bin per load); hist is 16-byte aligned.
__device__ void find_bin(const unsigned* hist, int nbins, unsigned remaining, int lane, int* bin_out,
                         unsigned* above_out) {
    const int per = nbins / 32;                       // 16 or 8 bins per lane, lane 0 the highest
    const int lo = nbins - per * (lane + 1);          // lane covers [lo, lo + per)
    unsigned v[16];
    const uint4* hv = reinterpret_cast<const uint4*>(hist + lo);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = q * 4 < per ? hv[q] : make_uint4(0u, 0u, 0u, 0u);
        v[4 * q] = u.x;
        v[4 * q + 1] = u.y;
        v[4 * q + 2] = u.z;
        v[4 * q + 3] = u.w;
    }
    unsigned mine = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mine += v[i];
    unsigned incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v2 = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v2;
    }
    const unsigned excl = incl - mine;
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining && excl < remaining);
    const int src = __ffs(hit) - 1;
    if (lane == src) {
        unsigned cum = excl;
        bool found = false;
#pragma unroll
        for (int i = 15; i >= 0; --i) {
            if (i < per && !found) {
                if (cum + v[i] >= remaining) {
                    *bin_out = lo + i;
                    *above_out = cum;
                    found = true;
                } else {
                    cum += v[i];
                }
            }
        }
    }
}

// Selection of chunk `chunk` of x (the CTA's 1,024 threads, one channel each);
// the chosen channels go to idx[chunk k ...] ascending and, when `sel_list` is
// given, to sel_list[0 .. count) in shared memory.  Returns the count.
__device__ int select_chunk(const __half* __restrict__ x, int K, int k, int32_t* __restrict__ idx, int chunk,
                            int* sel_list) {
    // one histogram and one (bin, count above) slot per pass, so no pass waits
    // for the one before it to be done reading
    __shared__ __align__(16) unsigned hist[512 + 256 + 256];
    __shared__ int s_bin[3];
    __shared__ unsigned s_above[3];
    __shared__ unsigned warp_cnt[kChunk / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int base = chunk * kChunk;
    const int len = min(kChunk, K - base);
    const int kk = min(k, len);
    const bool valid = t < len;
    unsigned key = 0;
    if (valid) {
        const unsigned short h = __half_as_ushort(x[base + t]);
        key = (static_cast<unsigned>(h & 0x7FFFu) << 10) | static_cast<unsigned>(kChunk - 1 - t);
    }
    // threshold = the kk-th largest key (every key when the chunk has <= k channels)
    unsigned thr = 0;
    if (kk < len) {
        unsigned prefix = 0, remaining = static_cast<unsigned>(kk);
        hist[t] = 0u;                                     // 1,024 counters, one per thread
        __syncthreads();
        // digits: key bits 24..16 (512 bins), 15..8, 7..0 (256 bins each)
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 16 : pass == 1 ? 8 : 0;
            const int nbins = pass == 0 ? 512 : 256;
            unsigned* h = hist + (pass == 0 ? 0 : pass == 1 ? 512 : 768);
            const bool cand = valid && (pass == 0 || (key >> (shift + 8)) == prefix);
            if (cand) atomicAdd(&h[(key >> shift) & (nbins - 1)], 1u);
            __syncthreads();
            if (warp == 0) find_bin(h, nbins, remaining, lane, &s_bin[pass], &s_above[pass]);
            __syncthreads();
            prefix = (pass == 0) ? static_cast<unsigned>(s_bin[pass])
                                 : ((prefix << 8) | static_cast<unsigned>(s_bin[pass]));
            remaining -= s_above[pass];
        }
        thr = prefix;   // all 25 bits: unique keys, so exactly kk keys are >= thr
    }
    const bool sel = valid && key >= thr;
    // ascending output: ballot prefix sum over the CTA
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    if (sel) {
        unsigned off = __popc(bal & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) off += warp_cnt[w];
        idx[static_cast<long long>(chunk) * k + off] = base + t;
        if (sel_list) sel_list[off] = base + t;
    }
    return kk;
}

__global__ void __launch_bounds__(kChunk) lbq_refine_select_kernel(const __half* __restrict__ x, int K, int k,
                                                                   int32_t* __restrict__ idx) {
    // launched with programmatic dependent launch: x may come from the kernel before
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    (void)select_chunk(x, K, k, idx, blockIdx.x, nullptr);
}

// Several selections in one launch (a layer's activation vectors): CTA b takes
// chunk b - chunk_ub[q] of problem q.  With a refinement blob, the CTA then
// prefetches the chosen columns' records into L2, so that the GEMV that applies
// them (lbq_gemv_grouped_refined, launched next) finds them there.
struct SelectProb {
    const __half* x;
    int32_t* idx;
    const uint8_t* refine;   // or nullptr
    int K, k;
    long long cb;            // refinement column bytes
};
struct SelectGroup {
    int count;
    int chunk_ub[LBQ_MAX_GROUP + 1];
    SelectProb p[LBQ_MAX_GROUP];
};

__global__ void __launch_bounds__(kChunk) lbq_refine_select_grouped_kernel(const __grid_constant__ SelectGroup g) {
    __shared__ int sel_list[lbq::kRefineMaxK];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int q = 0;
    while (q + 1 < g.count && g.chunk_ub[q + 1] <= static_cast<int>(blockIdx.x)) ++q;
    const SelectProb& pr = g.p[q];
    const int kk = select_chunk(pr.x, pr.K, pr.k, pr.idx, blockIdx.x - g.chunk_ub[q], sel_list);
    if (pr.refine) {
        __syncthreads();
        const int lines = static_cast<int>((pr.cb + 127) / 128);
        for (int i = threadIdx.x; i < kk * lines; i += kChunk) {
            const int c = sel_list[i / lines];
            const uint8_t* p = pr.refine + lbq::kRefineHeader + static_cast<long long>(c) * pr.cb + 128ll * (i % lines);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
}

// Header of a refinement blob: magic, version, shape (block 0 checks it).
__device__ __forceinline__ void check_refine_header(const uint8_t* blob, int N, int K, unsigned* err) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const unsigned* h = reinterpret_cast<const unsigned*>(blob);
        long long n_hdr, k_hdr;
        memcpy(&n_hdr, blob + 16, 8);
        memcpy(&k_hdr, blob + 24, 8);
        if (h[0] != 0x5251424Cu || h[1] != 0x43345746u || h[2] != lbq::kRefineVersion || n_hdr != N || k_hdr != K)
            atomicCAS(err, 0u, static_cast<unsigned>(LBQ_ERR_FORMAT));
    }
}

// y[row0 + n] += sum_j x[idx_j] C[row0 + n, idx_j] for the CTA's 256 rows.  The
// W warps take every W-th selected column; a lane owns one 32-bit nibble word
// (8 rows) of a group and accumulates x_i (q - z) s in FP32 ((q - z) s is exact
// in FP32); the warps' partial rows are added in warp order (deterministic) by
// threads 0..255.
template <int W>
__device__ __forceinline__ void apply_tile(const uint8_t* __restrict__ blob, int N, int K, const __half* x,
                                           const int32_t* idx, int nsel, void* y, int y_f32, unsigned* err,
                                           float (*part)[kApplyRows]) {
    constexpr int kApplyWarps = W;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * kApplyRows;
    const int g = (row0 >> 5) + (lane >> 2), wd = lane & 3;     // group and nibble word of this lane
    const bool rows_ok = g * 32 < N;
    const uint64_t cb = lbq::refine_column_bytes(N);
    if (warp < kApplyWarps) {
        float acc[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[b] = 0.f;
        // the warp's columns are j = warp + W c; their indices are loaded 32 at a
        // time (lane c holds column c's), then gathered four columns per round,
        // all loads of a round issued before any is used
        constexpr int kU = 4;
        for (int base = 0; base < nsel; base += kApplyWarps * 32) {
            const int jl = base + warp + kApplyWarps * lane;
            int mine = -1;
            if (jl < nsel) {
                mine = idx[jl];
                if (mine < 0 || mine >= K) {
                    atomicCAS(err, 0u, static_cast<unsigned>(LBQ_ERR_VALUE));
                    mine = -1;
                }
            }
            const int rest = nsel - base - warp;
            const int ncols = rest <= 0 ? 0 : min(32, (rest + kApplyWarps - 1) / kApplyWarps);
            for (int r0 = 0; r0 < ncols; r0 += kU) {
                int col_i[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = __shfl_sync(0xffffffffu, mine, (r0 + u) & 31);
                    col_i[u] = r0 + u < ncols ? c : -1;
                }
                float xi[kU], sc[kU], zf[kU];
                uint32_t word[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    xi[u] = 0.f;
                    sc[u] = 0.f;
                    zf[u] = 0.f;
                    word[u] = 0u;
                    if (col_i[u] >= 0 && rows_ok) {
                        const uint8_t* col = blob + lbq::kRefineHeader + static_cast<uint64_t>(col_i[u]) * cb;
                        xi[u] = __half2float(x[col_i[u]]);
                        word[u] = *reinterpret_cast<const uint32_t*>(col + g * 16 + wd * 4);
                        sc[u] = __half2float(*reinterpret_cast<const __half*>(col + N / 2 + g * 2));
                        const uint32_t zb = col[N / 2 + N / 16 + (g >> 1)];
                        zf[u] = static_cast<float>((g & 1) ? (zb >> 4) : (zb & 15u));
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const float lo = (static_cast<float>((word[u] >> (8 * b)) & 15u) - zf[u]) * sc[u];      // row 4 wd + b
                        const float hi = (static_cast<float>((word[u] >> (8 * b + 4)) & 15u) - zf[u]) * sc[u];  // row 16 + 4 wd + b
                        acc[b] = fmaf(lo, xi[u], acc[b]);
                        acc[4 + b] = fmaf(hi, xi[u], acc[4 + b]);
                    }
                }
            }
        }
        const int rbase = (lane >> 2) * 32 + 4 * wd;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            part[warp][rbase + b] = acc[b];
            part[warp][rbase + 16 + b] = acc[4 + b];
        }
    }
    __syncthreads();
    const int n = row0 + tid;
    if (tid < kApplyRows && n < N) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kApplyWarps; ++w) tot += part[w][tid];
        if (y_f32) {
            float* yf = static_cast<float*>(y);
            yf[n] = yf[n] + tot;
        } else {
            __half* yh = static_cast<__half*>(y);
            yh[n] = __float2half_rn(__half2float(yh[n]) + tot);
        }
    }
}

// W = 8 warps for short selections, 32 for long ones (224 columns after a
// K = 14336 projection: 18.2 -> 12.5 us measured)
template <int W>
__global__ void __launch_bounds__(W * 32) lbq_refine_apply_kernel(const uint8_t* __restrict__ blob, int N, int K,
                                                                  const __half* __restrict__ x,
                                                                  const int32_t* __restrict__ idx, int nsel, void* y,
                                                                  int y_f32, unsigned* err) {
    __shared__ float part[W][kApplyRows];
    // launched with programmatic dependent launch: idx, x and y come from the kernels before
    asm volatile("griddepcontrol.wait;" ::: "memory");
    check_refine_header(blob, N, K, err);
    apply_tile<W>(blob, N, K, x, idx, nsel, y, y_f32, err, part);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch with programmatic stream serialisation: the kernel may start while the
// previous one on the stream runs; it touches memory only after
// griddepcontrol.wait, so this is safe whatever that kernel wrote.
template <class... Args>
lbq_status launch_pdl(const void* fn, unsigned grid, unsigned block, void* stream, Args... args) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* ptrs[] = {static_cast<void*>(&args)...};
    if (cudaLaunchKernelExC(&cfg, fn, ptrs) != cudaSuccess) {
        (void)cudaGetLastError();
        return LBQ_ERR_CUDA;
    }
    return LBQ_OK;
}

// Device address of g_refine_idx_scratch for the current device, looked up
// once per device.
constexpr int kMaxDevicesNoAlloc = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_addr[kMaxDevicesNoAlloc] = {};

lbq_status refine_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LBQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevicesNoAlloc) return LBQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_refine_idx_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return LBQ_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_addr[dev];
    return LBQ_OK;
}

}  // namespace

extern "C" {

int64_t lbq_refine_selected_count(int64_t K, int32_t k) {
    if (K < 1 || K > lbq::kMaxK || k < 1 || k > lbq::kRefineMaxK) return 0;
    const int64_t full = K / kChunk, rest = K % kChunk;
    return full * k + (rest < k ? rest : k);
}

lbq_status lbq_refine_select(const void* x_f16, int64_t K, int32_t k, int32_t* idx, void* stream) {
    if (!x_f16 || !idx) return LBQ_ERR_NULL;
    if (K < 1 || K > lbq::kMaxK || k < 1 || k > lbq::kRefineMaxK) return LBQ_ERR_SHAPE;
    if (!aligned(x_f16, 2) || !aligned(idx, 4)) return LBQ_ERR_ALIGN;
    unsigned* err = nullptr;
    int sms = 0;
    const lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    const unsigned grid = static_cast<unsigned>((K + kChunk - 1) / kChunk);
    return launch_pdl(reinterpret_cast<const void*>(&lbq_refine_select_kernel), grid, kChunk, stream,
                      static_cast<const __half*>(x_f16), static_cast<int>(K), k, idx);
}

lbq_status lbq_refine_select_grouped(const lbq_refine_select_problem* problems, int32_t count, void* stream) {
    if (!problems) return LBQ_ERR_NULL;
    if (count < 1 || count > LBQ_MAX_GROUP) return LBQ_ERR_SHAPE;
    SelectGroup g;
    memset(&g, 0, sizeof(g));
    g.count = count;
    int chunks = 0;
    for (int i = 0; i < count; ++i) {
        const lbq_refine_select_problem& q = problems[i];
        if (!q.x || !q.idx) return LBQ_ERR_NULL;
        if (q.reserved != 0 || q.K < 1 || q.K > lbq::kMaxK || q.k < 1 || q.k > lbq::kRefineMaxK) return LBQ_ERR_SHAPE;
        if (q.refine && (q.N < 64 || q.N % 64 || q.N > INT32_MAX)) return LBQ_ERR_SHAPE;
        if (!aligned(q.x, 2) || !aligned(q.idx, 4) || (q.refine && !aligned(q.refine, 16))) return LBQ_ERR_ALIGN;
        SelectProb& p = g.p[i];
        p.x = static_cast<const __half*>(q.x);
        p.idx = q.idx;
        p.refine = static_cast<const uint8_t*>(q.refine);
        p.K = static_cast<int>(q.K);
        p.k = q.k;
        p.cb = q.refine ? static_cast<long long>(lbq_refine_packed_bytes(q.N, 1)) - lbq::kRefineHeader : 0;
        g.chunk_ub[i] = chunks;
        chunks += static_cast<int>((q.K + kChunk - 1) / kChunk);
    }
    g.chunk_ub[count] = chunks;
    unsigned* err = nullptr;
    int sms = 0;
    const lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    return launch_pdl(reinterpret_cast<const void*>(&lbq_refine_select_grouped_kernel), static_cast<unsigned>(chunks),
                      kChunk, stream, g);
}

lbq_status lbq_refine_apply(const void* refine, int64_t N, int64_t K, const void* x_f16, const int32_t* idx,
                            int32_t n_sel, void* y, lbq_dtype y_dtype, void* stream) {
    if (!refine || !x_f16 || !y || (n_sel > 0 && !idx)) return LBQ_ERR_NULL;
    if (N < 64 || N % 64 || N > INT32_MAX || K < 1 || K > lbq::kMaxK || n_sel < 0 || n_sel > K)
        return LBQ_ERR_SHAPE;
    if (y_dtype != LBQ_F16 && y_dtype != LBQ_F32) return LBQ_ERR_UNSUPPORTED;
    if (!aligned(refine, 16) || !aligned(x_f16, 2) || !aligned(y, y_dtype == LBQ_F32 ? 4 : 2) ||
        (idx && !aligned(idx, 4)))
        return LBQ_ERR_ALIGN;
    unsigned* err = nullptr;
    int sms = 0;
    const lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    const unsigned grid = static_cast<unsigned>((N + kApplyRows - 1) / kApplyRows);
    const bool wide = n_sel > kApplyWideFrom;
    return launch_pdl(wide ? reinterpret_cast<const void*>(&lbq_refine_apply_kernel<kApplyWarpsMax>)
                           : reinterpret_cast<const void*>(&lbq_refine_apply_kernel<8>),
                      grid, wide ? kApplyWarpsMax * 32 : 8 * 32, stream,
                      static_cast<const uint8_t*>(refine), static_cast<int>(N), static_cast<int>(K),
                      static_cast<const __half*>(x_f16), idx, static_cast<int>(n_sel), y, y_dtype == LBQ_F32 ? 1 : 0,
                      err);
}

lbq_status lbq_refine_noalloc(const void* refine, int64_t N, int64_t K, int32_t k, const void* x_f16, void* y,
                             lbq_dtype y_dtype, void* stream) {
    // every check of the two-call form first, so that an error leaves nothing enqueued
    if (!refine || !x_f16 || !y) return LBQ_ERR_NULL;
    if (N < 64 || N % 64 || N > INT32_MAX || K < 1 || K > lbq::kMaxK || k < 1 || k > lbq::kRefineMaxK)
        return LBQ_ERR_SHAPE;
    if (y_dtype != LBQ_F16 && y_dtype != LBQ_F32) return LBQ_ERR_UNSUPPORTED;
    if (!aligned(refine, 16) || !aligned(x_f16, 2) || !aligned(y, y_dtype == LBQ_F32 ? 4 : 2)) return LBQ_ERR_ALIGN;
    unsigned* err = nullptr;
    int sms = 0;
    lbq_status st = lbq::device_context(&err, &sms);
    if (st != LBQ_OK) return st;
    const int64_t n_sel = lbq_refine_selected_count(K, k);   // <= kNoAllocIdxMax for every valid (K, k)
    int32_t* idx = nullptr;
    st = refine_scratch(&idx);
    if (st != LBQ_OK) return st;
    // the selection writes every index the apply reads: nothing to clear
    st = lbq_refine_select(x_f16, K, k, idx, stream);
    if (st != LBQ_OK) return st;
    return lbq_refine_apply(refine, N, K, x_f16, idx, static_cast<int32_t>(n_sel), y, y_dtype, stream);
}

}  // extern "C"
