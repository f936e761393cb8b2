// Internal constants shared by the host (.cpp) and device (.cu) halves of liblbq.
#pragma once

#include <cstdint>

#include "lbq.h"

#define LBQ_VERSION_NUM 100          // 0.1.0
#define LBQ_FORMAT_VERSION_NUM 2

namespace lbq {

constexpr int64_t kMaxK = 65536;          // x of one row block must fit in shared memory
constexpr int32_t kMaxOutliers = 8192;    // gathered outlier activations live in shared memory
constexpr uint64_t kSectionAlign = 256;   // the record area and the index array start on this boundary
constexpr int kRowsPerBlock = 4;          // rows of a row block (one record row-block)
constexpr int kRecordGroups = 32;         // groups of 32 weights per dense record (1024 k)
constexpr int kOutlierCols = 256;         // outlier columns per full outlier record
constexpr int kOutlierColAlign = 8;       // the last outlier record's width is a multiple of this
constexpr int kMaxM = 64;                 // largest batch of the small-M entry point

uint16_t host_f64_to_f16(double v);

// Tensor-core 4-bit GEMM for 16 <= M <= 64 without outlier columns (lbq_mma.cu);
// err_word is the device error word of the library.
lbq_status launch_w4_mma(const void* packed, int64_t N, int64_t K, int M, const void* x, int64_t ldx, void* y,
                         int64_t ldy, bool y_f32, unsigned* err_word, int sms, int max_smem, void* stream,
                         uint32_t flags);
double host_f16_to_f64(uint16_t h);

}  // namespace lbq
