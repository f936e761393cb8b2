// Internal constants shared by the host (.cpp) and device (.cu) halves of liblbq.
#pragma once

#include <cstdint>

#include "lbq.h"

#define LBQ_VERSION_NUM 100          // 0.1.0
#define LBQ_FORMAT_VERSION_NUM 2

#ifdef __CUDACC__
#define LBQ_HOST_DEVICE __host__ __device__
#else
#define LBQ_HOST_DEVICE
#endif

namespace lbq {

constexpr int64_t kMaxK = 65536;          // x of one row block must fit in shared memory
constexpr int32_t kMaxOutliers = 8192;    // gathered outlier activations live in shared memory
constexpr uint64_t kSectionAlign = 256;   // the record area and the index array start on this boundary
constexpr int kRowsPerBlock = 4;          // rows of a row block (one record row-block)
constexpr int kRecordGroups = 32;         // groups of 32 weights per dense record (1024 k)
constexpr int kOutlierCols = 256;         // outlier columns per full outlier record
constexpr int kOutlierColAlign = 8;       // the last outlier record's width is a multiple of this
constexpr int kMaxM = 64;                 // largest batch of the small-M entry point

// selective refinement blob (lbq_pack_refine / lbq_refine_apply): 64-byte
// header, then one record per input channel of N/2 nibble bytes, N/32 FP16
// scales and N/64 zero-point bytes, padded to 16 bytes
constexpr uint32_t kRefineHeader = 64;
constexpr uint32_t kRefineVersion = 1;
constexpr int kRefineChunk = 1024;        // channels per selection chunk
constexpr int kRefineMaxK = 256;          // largest channels-per-chunk budget
LBQ_HOST_DEVICE inline uint64_t refine_column_bytes(int64_t N) {
    return (static_cast<uint64_t>(N / 2 + N / 16 + N / 64) + 15) / 16 * 16;
}

// The device error word of the library and the SM count of the current device
// (lbq_gemv.cu); LBQ_ERR_UNSUPPORTED without an sm_103a device.
lbq_status device_context(unsigned** err_word, int* sms);

uint16_t host_f64_to_f16(double v);

// Tensor-core 4-bit GEMM for 16 <= M <= 64, outlier columns added in its
// epilogue (lbq_mma_w4.cu); err_word is the device error word of the library.
lbq_status launch_w4_mma(const void* packed, int64_t N, int64_t K, int32_t n_out, int M, const void* x, int64_t ldx,
                         void* y, int64_t ldy, bool y_f32, unsigned* err_word, int sms, int max_smem, void* stream,
                         uint32_t flags);
// Tensor-core 2-bit codebook GEMM for 16 <= M <= 64 with its exact FP16
// outlier columns (lbq_mma.cu).  One launch per slab of 256-row tiles; with
// `launches` set it only adds the number of launches.  LBQ_ERR_SHAPE when the
// problem does not fit.
lbq_status launch_w2_mma(const void* packed, int64_t N, int64_t K, int32_t n_out, int M, const void* x, int64_t ldx,
                         void* y, int64_t ldy, bool y_f32, unsigned* err_word, int max_smem, void* stream,
                         uint32_t flags, int* launches);
double host_f16_to_f64(uint16_t h);

// Work split of the tensor-core kernels: T tiles of Ut stages each are cut into
// G clusters of consecutive tiles (cluster c: tiles [t0, t1)), and a cluster's
// units = (t1 - t0) x Ut stages into C contiguous ranges (rank r: [u0, u1)).
// 32-bit arithmetic (the planner keeps T x Ut x C below 2^31): the kernels
// evaluate these in their prologue and epilogue, where 64-bit divisions cost
// microseconds.
LBQ_HOST_DEVICE inline void cluster_tiles(int T, int G, int c, int* t0, int* t1) {
    *t0 = T * c / G;
    *t1 = T * (c + 1) / G;
}
LBQ_HOST_DEVICE inline void rank_range(int units, int C, int r, int* u0, int* u1) {
    *u0 = units * r / C;
    *u1 = units * (r + 1) / C;
}
// The rank whose range holds stage u (ranges are contiguous and ascending).
LBQ_HOST_DEVICE inline int rank_of(int units, int C, int u) {
    int r = (u * C) / (units > 0 ? units : 1);
    if (r > C - 1) r = C - 1;
    while (r > 0 && units * r / C > u) --r;
    while (r + 1 < C && units * (r + 1) / C <= u) ++r;
    return r;
}
// The cluster size C and cluster count G that give the fewest stages to the
// busiest CTA, every CTA's range spanning at most `bands` tiles; active[c] is
// the number of clusters of size c that fit the device at once (0: none).
// False when no cluster size fits (lbq_mma.cu).
bool mma_plan(int T, int Ut, int bands, const int* active, int* C_out, int* G_out, int* load_out);

}  // namespace lbq
