// Host side of liblbq: blob layout, FP16 rounding, outlier selection and the
// 4-bit / 2-bit quantise-and-pack routines.  Pure C++17, no CUDA.
//
// Must be compiled with -ffp-contract=off and without fast-math: the packed
// bytes are defined by an exact FP64 recipe (sequential sums, IEEE division
// and square root, round-half-to-even), so that two independent
// implementations of the same formulas produce identical bytes.

#include <algorithm>
#include <atomic>
#include <cfenv>
#include <cmath>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

#include "lbq.h"
#include "lbq_internal.h"

namespace {

constexpr int kGroup = 32;
constexpr double kScaleFloor = 1e-8;    // SPECTRA 3.4: s = max(range / 15, 1e-8)
constexpr double kOlsEps = 1e-8;        // otf-llm 3: OLS denominator epsilon (value is a reading)
constexpr uint32_t kHeaderBytes = 128;
// part offsets inside a dense record (4 rows x 32 groups)
constexpr uint64_t kW4ScaleOff = 4 * 32 * 16;                 // 2048
constexpr uint64_t kW4ZeroOff = kW4ScaleOff + 4 * 32 * 2;     // 2304
constexpr uint64_t kW2SOff = 4 * 32 * 8;                      // 1024
constexpr uint64_t kW2ZOff = kW2SOff + 4 * 32 * 2;            // 1280

// otf-llm section 2 codebook, rounded once to FP16 (bit patterns and values)
constexpr double kCodebookDecimal[4] = {-1.52, -0.45, 0.45, 1.52};

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Round a double to the nearest IEEE binary16 value, ties to even, computed
// from the double's bit pattern (no intermediate float, so no double rounding).
uint16_t f64_to_f16_bits(double v) {
    uint64_t b;
    std::memcpy(&b, &v, 8);
    const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
    const int exp = static_cast<int>((b >> 52) & 0x7FF);
    uint64_t man = b & ((uint64_t(1) << 52) - 1);
    if (exp == 0x7FF) return sign | (man ? 0x7E00 : 0x7C00);
    if (exp == 0 && man == 0) return sign;
    // value = 1.man * 2^(exp-1023) for normal doubles (double subnormals are far
    // below the FP16 range and round to zero below)
    const int e = exp - 1023;
    if (exp == 0) return sign;                   // |v| < 2^-1022: rounds to 0
    if (e > 15) return sign | 0x7C00;            // >= 2^16: overflow
    uint64_t sig = man | (uint64_t(1) << 52);    // 53-bit significand
    int shift;                                   // bits to drop from sig
    uint16_t exp_field;
    if (e >= -14) {                              // FP16 normal range
        shift = 52 - 10;
        exp_field = static_cast<uint16_t>(e + 15);
    } else {                                     // FP16 subnormal: unit 2^-24
        shift = 52 - 10 + (-14 - e);
        exp_field = 0;
        if (shift > 63) return sign;             // far below 2^-25
    }
    uint64_t kept = sig >> shift;
    const uint64_t rem = sig & ((uint64_t(1) << shift) - 1);
    const uint64_t half = uint64_t(1) << (shift - 1);
    if (rem > half || (rem == half && (kept & 1))) kept += 1;
    uint32_t out;
    if (exp_field == 0) {
        out = static_cast<uint32_t>(kept);       // may carry into 0x400 = min normal
    } else {
        // kept in [2^10, 2^11]; a carry to 2^11 bumps the exponent
        if (kept == (uint64_t(1) << 11)) {
            kept >>= 1;
            exp_field += 1;
        }
        if (exp_field >= 31) return sign | 0x7C00;
        out = (uint32_t(exp_field) << 10) | static_cast<uint32_t>(kept & 0x3FF);
    }
    return static_cast<uint16_t>(sign | out);
}

double f16_bits_to_f64(uint16_t h) {
    const int sign = (h & 0x8000) ? -1 : 1;
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    if (e == 0) return sign * std::ldexp(static_cast<double>(m), -24);
    if (e == 31) return m ? std::nan("") : sign * HUGE_VAL;
    return sign * std::ldexp(static_cast<double>(1024 + m), e - 25);
}

struct Codebook {
    uint16_t bits[4];
    double val[4];
    Codebook() {
        for (int c = 0; c < 4; ++c) {
            bits[c] = f64_to_f16_bits(kCodebookDecimal[c]);
            val[c] = f16_bits_to_f64(bits[c]);
        }
    }
};
const Codebook& codebook() {
    static const Codebook cb;
    return cb;
}

bool shape_ok(int64_t N, int64_t K, int32_t n_out) {
    return N >= 1 && N <= INT32_MAX && K >= 64 && K <= lbq::kMaxK && K % 64 == 0 && n_out >= 0 &&
           n_out <= K && n_out <= lbq::kMaxOutliers;
}

// Run fn(begin, end) over [0, n) on up to hardware_concurrency threads.
template <class F>
void parallel_for(int64_t n, F fn) {
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, 64));
    nt = std::min<int64_t>(nt, std::max<int64_t>(1, n / 16));
    if (nt <= 1) {
        fn(int64_t(0), n);
        return;
    }
    std::vector<std::thread> th;
    const int64_t chunk = (n + nt - 1) / nt;
    for (int64_t t = 0; t < nt; ++t) {
        const int64_t b = t * chunk, e = std::min(n, b + chunk);
        if (b >= e) break;
        th.emplace_back([=] { fn(b, e); });
    }
    for (auto& t : th) t.join();
}

bool all_finite(const float* W, int64_t count) {
    std::atomic<bool> ok{true};
    parallel_for(count, [&](int64_t b, int64_t e) {
        for (int64_t i = b; i < e; ++i)
            if (!std::isfinite(W[i])) {
                ok = false;
                return;
            }
    });
    return ok;
}

lbq_status check_idx(const int32_t* idx, int32_t n_out, int64_t K) {
    if (n_out > 0 && !idx) return LBQ_ERR_NULL;
    for (int32_t j = 0; j < n_out; ++j) {
        if (idx[j] < 0 || idx[j] >= K) return LBQ_ERR_OUTLIER_IDX;
        if (j > 0 && idx[j] <= idx[j - 1]) return LBQ_ERR_OUTLIER_IDX;
    }
    return LBQ_OK;
}

// ||W[:, j]||_2 in FP64, the squares accumulated row by row in order.
std::vector<double> column_norms(const float* W, int64_t N, int64_t K) {
    std::vector<double> acc(static_cast<size_t>(K), 0.0);
    parallel_for(K, [&](int64_t b, int64_t e) {
        for (int64_t n = 0; n < N; ++n) {
            const float* row = W + n * K;
            for (int64_t j = b; j < e; ++j) {
                const double w = row[j];
                const double sq = w * w;
                acc[j] = acc[j] + sq;
            }
        }
    });
    for (auto& a : acc) a = std::sqrt(a);
    return acc;
}

// n largest scores, ties to the lower index; returned ascending.
std::vector<int32_t> top_n(const std::vector<double>& score, int64_t n) {
    std::vector<int32_t> order(score.size());
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        if (score[a] != score[b]) return score[a] > score[b];
        return a < b;
    });
    order.resize(static_cast<size_t>(n));
    std::sort(order.begin(), order.end());
    return order;
}

lbq_status emit_indices(const std::vector<int32_t>& sel, int32_t* idx, int32_t cap, int32_t* n_out) {
    *n_out = static_cast<int32_t>(sel.size());
    if (static_cast<int64_t>(sel.size()) > cap) return LBQ_ERR_BUFFER_TOO_SMALL;
    if (!sel.empty() && !idx) return LBQ_ERR_NULL;
    std::copy(sel.begin(), sel.end(), idx);
    return LBQ_OK;
}

void write_header(uint8_t* dst, const char magic[8], int64_t N, int64_t K, int32_t n_out,
                  const lbq_layout& L) {
    std::memset(dst, 0, kHeaderBytes);
    std::memcpy(dst, magic, 8);
    const uint32_t version = LBQ_FORMAT_VERSION_NUM, hbytes = kHeaderBytes, group = kGroup;
    std::memcpy(dst + 8, &version, 4);
    std::memcpy(dst + 12, &hbytes, 4);
    std::memcpy(dst + 16, &N, 8);
    std::memcpy(dst + 24, &K, 8);
    std::memcpy(dst + 32, &n_out, 4);
    std::memcpy(dst + 36, &group, 4);
    std::memcpy(dst + 40, &L.total_bytes, 8);
    const uint64_t f[7] = {L.area_offset, L.row_block_bytes, L.record_bytes, L.records,
                           L.outlier_record_bytes, L.outlier_records, L.idx_offset};
    std::memcpy(dst + 48, f, sizeof(f));
}

// SPECTRA 3.4 / App. A Prop. 2 on one group of 32 values, in FP64 with the
// unrounded scale: s = max((wmax - wmin) / 15, 1e-8), z = clamp(round(-wmin / s)),
// q = clamp(round(w / s + z)), rounding half to even.
void quantise_group_w4(const double (&w)[kGroup], uint8_t (&q)[kGroup], double* s_out, uint8_t* z_out) {
    double wmin = HUGE_VAL, wmax = -HUGE_VAL;
    for (int k = 0; k < kGroup; ++k) {
        wmin = std::min(wmin, w[k]);
        wmax = std::max(wmax, w[k]);
    }
    const double s = std::max((wmax - wmin) / 15.0, kScaleFloor);
    const double z = std::min(std::max(std::nearbyint(-wmin / s), 0.0), 15.0);
    for (int k = 0; k < kGroup; ++k) {
        double t = w[k] / s;
        t = t + z;
        q[k] = static_cast<uint8_t>(std::min(std::max(std::nearbyint(t), 0.0), 15.0));
    }
    *s_out = s;
    *z_out = static_cast<uint8_t>(z);
}

// Byte offset of (row n, group g) inside the blob's record area: the record of
// row block n/4 and group block g/32, plus the row-major (row, group) index.
struct RecordAddr {
    uint64_t rec;     // start of the record
    int slot;         // (row in block) * 32 + (group in record)
};
inline RecordAddr record_addr(const lbq_layout& L, int64_t n, int64_t g) {
    RecordAddr a;
    a.rec = L.area_offset + uint64_t(n / lbq::kRowsPerBlock) * L.row_block_bytes +
            uint64_t(g / lbq::kRecordGroups) * L.record_bytes;
    a.slot = int(n % lbq::kRowsPerBlock) * lbq::kRecordGroups + int(g % lbq::kRecordGroups);
    return a;
}

// Shared front matter of both packers: validation, header, outlier sections.
// Returns a per-row mask of outlier columns through is_out.
lbq_status pack_common(lbq_kind kind, const float* W, int64_t N, int64_t K, const int32_t* idx,
                       int32_t n_out, void* dst, size_t dst_bytes, lbq_layout* L,
                       std::vector<uint8_t>* is_out) {
    if (!W || !dst) return LBQ_ERR_NULL;
    if (!shape_ok(N, K, n_out)) return LBQ_ERR_SHAPE;
    lbq_status st = check_idx(idx, n_out, K);
    if (st != LBQ_OK) return st;
    st = lbq_blob_layout(kind, N, K, n_out, L);
    if (st != LBQ_OK) return st;
    if (dst_bytes < L->total_bytes) return LBQ_ERR_BUFFER_TOO_SMALL;
    if (!all_finite(W, N * K)) return LBQ_ERR_VALUE;
    uint8_t* out = static_cast<uint8_t*>(dst);
    std::memset(out, 0, L->total_bytes);
    write_header(out, kind == LBQ_KIND_W4 ? "LBQW4G32" : "LBQW2C32", N, K, n_out, *L);
    is_out->assign(static_cast<size_t>(K), 0);
    for (int32_t j = 0; j < n_out; ++j) (*is_out)[idx[j]] = 1;
    if (n_out > 0) {
        std::memcpy(out + L->idx_offset, idx, sizeof(int32_t) * n_out);
        // outlier records follow the dense records of each row block
        parallel_for(N, [&](int64_t b, int64_t e) {
            for (int64_t n = b; n < e; ++n) {
                const uint64_t base = L->area_offset + uint64_t(n / lbq::kRowsPerBlock) * L->row_block_bytes +
                                      L->records * L->record_bytes;
                const int r = int(n % lbq::kRowsPerBlock);
                for (int32_t j = 0; j < n_out; ++j) {
                    const int32_t rec = j / lbq::kOutlierCols;
                    const uint64_t width = std::min<uint64_t>(
                        lbq::kOutlierCols, round_up(uint64_t(n_out), lbq::kOutlierColAlign) - uint64_t(rec) * lbq::kOutlierCols);
                    const uint64_t off = base + uint64_t(rec) * L->outlier_record_bytes +
                                         (uint64_t(r) * width + uint64_t(j % lbq::kOutlierCols)) * 2;
                    const uint16_t h = f64_to_f16_bits(W[n * K + idx[j]]);
                    std::memcpy(out + off, &h, 2);
                }
            }
        });
    }
    return LBQ_OK;
}

}  // namespace

namespace lbq {
uint16_t host_f64_to_f16(double v) { return f64_to_f16_bits(v); }
double host_f16_to_f64(uint16_t h) { return f16_bits_to_f64(h); }
}  // namespace lbq

extern "C" {

int lbq_version(void) { return LBQ_VERSION_NUM; }
int lbq_format_version(void) { return LBQ_FORMAT_VERSION_NUM; }

const char* lbq_status_string(lbq_status s) {
    switch (s) {
        case LBQ_OK: return "LBQ_OK";
        case LBQ_ERR_NULL: return "LBQ_ERR_NULL: a required pointer is NULL";
        case LBQ_ERR_SHAPE: return "LBQ_ERR_SHAPE: N, K, M, n_out or a leading dimension out of range";
        case LBQ_ERR_ALIGN: return "LBQ_ERR_ALIGN: pointer or leading dimension misaligned";
        case LBQ_ERR_OUTLIER_IDX: return "LBQ_ERR_OUTLIER_IDX: outlier indices not ascending or out of range";
        case LBQ_ERR_BUFFER_TOO_SMALL: return "LBQ_ERR_BUFFER_TOO_SMALL: destination smaller than required";
        case LBQ_ERR_FORMAT: return "LBQ_ERR_FORMAT: blob header does not match the call";
        case LBQ_ERR_CUDA: return "LBQ_ERR_CUDA: CUDA runtime or launch error";
        case LBQ_ERR_TIMEOUT: return "LBQ_ERR_TIMEOUT: a bounded in-kernel wait gave up";
        case LBQ_ERR_VALUE: return "LBQ_ERR_VALUE: non-finite input or argument out of range";
        case LBQ_ERR_UNSUPPORTED: return "LBQ_ERR_UNSUPPORTED: unsupported device or argument";
    }
    return "LBQ_ERR_UNKNOWN";
}

lbq_status lbq_blob_layout(lbq_kind kind, int64_t N, int64_t K, int32_t n_out, lbq_layout* out) {
    if (!out) return LBQ_ERR_NULL;
    if (!shape_ok(N, K, n_out)) return LBQ_ERR_SHAPE;
    uint64_t per_row;   // bytes of one row of a record: packed + scale/S + zero/Z for 32 groups
    if (kind == LBQ_KIND_W4)
        per_row = 16 * lbq::kRecordGroups + 2 * lbq::kRecordGroups + lbq::kRecordGroups / 2;
    else if (kind == LBQ_KIND_W2CB)
        per_row = 8 * lbq::kRecordGroups + 2 * lbq::kRecordGroups + 2 * lbq::kRecordGroups;
    else
        return LBQ_ERR_UNSUPPORTED;
    const uint64_t group_k = uint64_t(lbq::kRecordGroups) * kGroup;
    out->area_offset = lbq::kSectionAlign;
    out->record_bytes = lbq::kRowsPerBlock * per_row;
    out->records = (uint64_t(K) + group_k - 1) / group_k;
    out->outlier_record_bytes = n_out > 0 ? uint64_t(lbq::kRowsPerBlock) * lbq::kOutlierCols * 2 : 0;
    out->outlier_records = (uint64_t(n_out) + lbq::kOutlierCols - 1) / lbq::kOutlierCols;
    // the last outlier record holds the remaining columns rounded up to a multiple of 8
    const uint64_t out_cols = round_up(uint64_t(n_out), lbq::kOutlierColAlign);
    out->row_block_bytes = out->records * out->record_bytes + uint64_t(lbq::kRowsPerBlock) * 2 * out_cols;
    const uint64_t n_rb = (uint64_t(N) + lbq::kRowsPerBlock - 1) / lbq::kRowsPerBlock;
    out->idx_offset = round_up(out->area_offset + n_rb * out->row_block_bytes, lbq::kSectionAlign);
    out->total_bytes = round_up(out->idx_offset + 4ull * n_out, lbq::kSectionAlign);
    return LBQ_OK;
}

size_t lbq_w4_packed_bytes(int64_t N, int64_t K, int32_t n_out) {
    lbq_layout L;
    return lbq_blob_layout(LBQ_KIND_W4, N, K, n_out, &L) == LBQ_OK ? L.total_bytes : 0;
}

size_t lbq_w2cb_packed_bytes(int64_t N, int64_t K, int32_t n_out) {
    lbq_layout L;
    return lbq_blob_layout(LBQ_KIND_W2CB, N, K, n_out, &L) == LBQ_OK ? L.total_bytes : 0;
}

lbq_status lbq_select_outliers_w4(const float* W, int64_t N, int64_t K, int32_t* idx, int32_t cap,
                                  int32_t* n_out) {
    if (!W || !n_out) return LBQ_ERR_NULL;
    if (!shape_ok(N, K, 0)) return LBQ_ERR_SHAPE;
    if (!all_finite(W, N * K)) return LBQ_ERR_VALUE;
    const std::vector<double> S = column_norms(W, N, K);
    // population kurtosis of the saliencies (SPECTRA Proposition 1)
    double sum = S[0];
    for (int64_t j = 1; j < K; ++j) sum = sum + S[j];
    const double mu = sum / static_cast<double>(K);
    std::vector<double> d(static_cast<size_t>(K));
    for (int64_t j = 0; j < K; ++j) d[j] = S[j] - mu;
    double ss = d[0] * d[0];
    for (int64_t j = 1; j < K; ++j) {
        const double sq = d[j] * d[j];
        ss = ss + sq;
    }
    const double sigma = std::sqrt(ss / static_cast<double>(K));
    double kappa = 0.0;
    if (sigma != 0.0) {
        double s4 = 0.0;
        for (int64_t j = 0; j < K; ++j) {
            const double z = d[j] / sigma;
            const double z2 = z * z;
            const double z4 = z2 * z2;
            s4 = (j == 0) ? z4 : s4 + z4;
        }
        kappa = s4 / static_cast<double>(K);
    }
    // SPECTRA 3.3: r = clamp(r_base (1 + 0.15 ln(1 + max(0, kappa - 3))), 0.005, 0.03)
    double r = 0.01 * (1.0 + 0.15 * std::log(1.0 + std::max(0.0, kappa - 3.0)));
    r = std::min(std::max(r, 0.005), 0.03);
    const int64_t count = static_cast<int64_t>(std::floor(r * static_cast<double>(K)));
    return emit_indices(top_n(S, count), idx, cap, n_out);
}

lbq_status lbq_select_outliers_impact(const float* W, int64_t N, int64_t K, const uint16_t* Xprof_f16,
                                      int32_t P, double frac, int32_t* idx, int32_t cap,
                                      int32_t* n_out) {
    if (!W || !Xprof_f16 || !n_out) return LBQ_ERR_NULL;
    if (!shape_ok(N, K, 0) || P < 1) return LBQ_ERR_SHAPE;
    if (!(frac >= 0.0 && frac <= 1.0)) return LBQ_ERR_VALUE;
    if (!all_finite(W, N * K)) return LBQ_ERR_VALUE;
    std::vector<double> S = column_norms(W, N, K);
    // otf-llm section 4: I_c = ||W[:,c]||_2 * mean_p |x_{p,c}|
    std::vector<double> acc(static_cast<size_t>(K), 0.0);
    for (int32_t p = 0; p < P; ++p)
        for (int64_t c = 0; c < K; ++c) {
            const double a = std::fabs(f16_bits_to_f64(Xprof_f16[int64_t(p) * K + c]));
            if (!std::isfinite(a)) return LBQ_ERR_VALUE;
            acc[c] = acc[c] + a;
        }
    for (int64_t c = 0; c < K; ++c) S[c] = S[c] * (acc[c] / static_cast<double>(P));
    const int64_t count = static_cast<int64_t>(std::floor(frac * static_cast<double>(K)));
    return emit_indices(top_n(S, count), idx, cap, n_out);
}

lbq_status lbq_pack_w4(const float* W, int64_t N, int64_t K, const int32_t* idx, int32_t n_out,
                       void* dst, size_t dst_bytes) {
    lbq_layout L;
    std::vector<uint8_t> is_out;
    lbq_status st = pack_common(LBQ_KIND_W4, W, N, K, idx, n_out, dst, dst_bytes, &L, &is_out);
    if (st != LBQ_OK) return st;
    uint8_t* out = static_cast<uint8_t*>(dst);
    const int64_t ng = K / kGroup;
    parallel_for(N, [&](int64_t b, int64_t e) {
        double w[kGroup];
        uint8_t q[kGroup];
        for (int64_t n = b; n < e; ++n) {
            for (int64_t g = 0; g < ng; ++g) {
                const RecordAddr ra = record_addr(L, n, g);
                for (int k = 0; k < kGroup; ++k) {
                    const int64_t col = g * kGroup + k;
                    w[k] = is_out[col] ? 0.0 : static_cast<double>(W[n * K + col]);
                }
                double s;
                uint8_t zi;
                quantise_group_w4(w, q, &s, &zi);
                uint8_t* qdst = out + ra.rec + uint64_t(ra.slot) * 16;
                for (int k = 0; k < 16; ++k) qdst[k] = static_cast<uint8_t>(q[k] | (q[k + 16] << 4));
                const uint16_t sh = f64_to_f16_bits(s);
                std::memcpy(out + ra.rec + kW4ScaleOff + uint64_t(ra.slot) * 2, &sh, 2);
                uint8_t* zdst = out + ra.rec + kW4ZeroOff + (ra.slot >> 1);   // (row * 32 + group) / 2
                if (g % 2 == 0)
                    *zdst = zi;
                else
                    *zdst = static_cast<uint8_t>(*zdst | (zi << 4));
            }
        }
    });
    return LBQ_OK;
}

lbq_status lbq_pack_w2cb(const float* W, int64_t N, int64_t K, const int32_t* idx, int32_t n_out,
                         void* dst, size_t dst_bytes) {
    lbq_layout L;
    std::vector<uint8_t> is_out;
    lbq_status st = pack_common(LBQ_KIND_W2CB, W, N, K, idx, n_out, dst, dst_bytes, &L, &is_out);
    if (st != LBQ_OK) return st;
    uint8_t* out = static_cast<uint8_t*>(dst);
    const Codebook& cb = codebook();
    const int64_t ng = K / kGroup;
    parallel_for(N, [&](int64_t b, int64_t e) {
        double w[kGroup], d[kGroup], cq[kGroup];
        uint8_t q[kGroup];
        for (int64_t n = b; n < e; ++n) {
            for (int64_t g = 0; g < ng; ++g) {
                const RecordAddr ra = record_addr(L, n, g);
                for (int k = 0; k < kGroup; ++k) {
                    const int64_t col = g * kGroup + k;
                    w[k] = is_out[col] ? 0.0 : static_cast<double>(W[n * K + col]);
                }
                // standardise by the group mean and population standard deviation
                double sum = w[0];
                for (int k = 1; k < kGroup; ++k) sum = sum + w[k];
                const double mu = sum / kGroup;
                for (int k = 0; k < kGroup; ++k) d[k] = w[k] - mu;
                double ss = d[0] * d[0];
                for (int k = 1; k < kGroup; ++k) {
                    const double sq = d[k] * d[k];
                    ss = ss + sq;
                }
                const double sigma = std::sqrt(ss / kGroup);
                for (int k = 0; k < kGroup; ++k) {
                    const double u = sigma > 0.0 ? d[k] / sigma : 0.0;
                    int best = 0;
                    double bd = std::fabs(u - cb.val[0]);
                    for (int c = 1; c < 4; ++c) {
                        const double dc = std::fabs(u - cb.val[c]);
                        if (dc < bd) {
                            bd = dc;
                            best = c;
                        }
                    }
                    q[k] = static_cast<uint8_t>(best);
                    cq[k] = cb.val[best];
                }
                // otf-llm section 3: closed-form least squares for (S, Z)
                double csum = cq[0];
                for (int k = 1; k < kGroup; ++k) csum = csum + cq[k];
                const double cbar = csum / kGroup;
                double num = 0.0, den = 0.0;
                for (int k = 0; k < kGroup; ++k) {
                    const double dw = w[k] - mu;
                    const double dc = cq[k] - cbar;
                    const double p = dw * dc;
                    const double p2 = dc * dc;
                    num = (k == 0) ? p : num + p;
                    den = (k == 0) ? p2 : den + p2;
                }
                const double S = num / (den + kOlsEps);
                const double SZ = S * cbar;
                const double Z = mu - SZ;
                const uint16_t Sh = f64_to_f16_bits(S), Zh = f64_to_f16_bits(Z);
                std::memcpy(out + ra.rec + kW2SOff + uint64_t(ra.slot) * 2, &Sh, 2);
                std::memcpy(out + ra.rec + kW2ZOff + uint64_t(ra.slot) * 2, &Zh, 2);
                uint8_t* cdst = out + ra.rec + uint64_t(ra.slot) * 8;
                for (int i = 0; i < kGroup / 4; ++i)
                    cdst[i] = static_cast<uint8_t>(q[4 * i] | (q[4 * i + 1] << 2) | (q[4 * i + 2] << 4) |
                                                   (q[4 * i + 3] << 6));
            }
        }
    });
    return LBQ_OK;
}

// ------------------------------------------------------- selective refinement

size_t lbq_refine_packed_bytes(int64_t N, int64_t K) {
    if (N < 64 || N % 64 || N > INT32_MAX || K < 1 || K > lbq::kMaxK) return 0;
    return lbq::kRefineHeader + static_cast<size_t>(K) * lbq::refine_column_bytes(N);
}

lbq_status lbq_pack_refine(const float* R, int64_t N, int64_t K, void* dst, size_t dst_bytes) {
    if (!R || !dst) return LBQ_ERR_NULL;
    const size_t total = lbq_refine_packed_bytes(N, K);
    if (total == 0) return LBQ_ERR_SHAPE;
    if (dst_bytes < total) return LBQ_ERR_BUFFER_TOO_SMALL;
    if (!all_finite(R, N * K)) return LBQ_ERR_VALUE;
    uint8_t* out = static_cast<uint8_t*>(dst);
    std::memset(out, 0, total);
    const uint64_t cb = lbq::refine_column_bytes(N);
    std::memcpy(out, "LBQRFW4C", 8);
    const uint32_t version = lbq::kRefineVersion, hbytes = lbq::kRefineHeader, group = kGroup,
                   cb32 = static_cast<uint32_t>(cb);
    const uint64_t tot = total;
    std::memcpy(out + 8, &version, 4);
    std::memcpy(out + 12, &hbytes, 4);
    std::memcpy(out + 16, &N, 8);
    std::memcpy(out + 24, &K, 8);
    std::memcpy(out + 32, &group, 4);
    std::memcpy(out + 36, &cb32, 4);
    std::memcpy(out + 40, &tot, 8);
    const int64_t ng = N / kGroup;
    parallel_for(K, [&](int64_t b, int64_t e) {
        double w[kGroup];
        uint8_t q[kGroup];
        for (int64_t i = b; i < e; ++i) {
            uint8_t* col = out + lbq::kRefineHeader + uint64_t(i) * cb;
            for (int64_t g = 0; g < ng; ++g) {
                for (int k = 0; k < kGroup; ++k) w[k] = static_cast<double>(R[(g * kGroup + k) * K + i]);
                double s;
                uint8_t z;
                quantise_group_w4(w, q, &s, &z);
                for (int k = 0; k < 16; ++k) col[g * 16 + k] = static_cast<uint8_t>(q[k] | (q[k + 16] << 4));
                const uint16_t sh = f64_to_f16_bits(s);
                std::memcpy(col + N / 2 + g * 2, &sh, 2);
                uint8_t* zb = col + N / 2 + N / 16 + g / 2;
                *zb = (g % 2 == 0) ? z : static_cast<uint8_t>(*zb | (z << 4));
            }
        }
    });
    return LBQ_OK;
}

lbq_status lbq_dequant_host(const void* packed, size_t packed_bytes, float* W_hat) {
    if (!packed || !W_hat) return LBQ_ERR_NULL;
    const uint8_t* in = static_cast<const uint8_t*>(packed);
    if (packed_bytes < kHeaderBytes) return LBQ_ERR_BUFFER_TOO_SMALL;
    const bool w4 = std::memcmp(in, "LBQW4G32", 8) == 0, w2 = std::memcmp(in, "LBQW2C32", 8) == 0;
    uint32_t version;
    std::memcpy(&version, in + 8, 4);
    if ((!w4 && !w2) || version != LBQ_FORMAT_VERSION_NUM) return LBQ_ERR_FORMAT;
    int64_t N, K;
    int32_t n_out;
    std::memcpy(&N, in + 16, 8);
    std::memcpy(&K, in + 24, 8);
    std::memcpy(&n_out, in + 32, 4);
    if (!shape_ok(N, K, n_out)) return LBQ_ERR_FORMAT;
    lbq_layout L;
    lbq_status st = lbq_blob_layout(w4 ? LBQ_KIND_W4 : LBQ_KIND_W2CB, N, K, n_out, &L);
    if (st != LBQ_OK) return st;
    if (packed_bytes < L.total_bytes) return LBQ_ERR_BUFFER_TOO_SMALL;
    std::vector<int32_t> idx(static_cast<size_t>(n_out));
    if (n_out > 0) std::memcpy(idx.data(), in + L.idx_offset, sizeof(int32_t) * n_out);
    st = check_idx(idx.data(), n_out, K);
    if (st != LBQ_OK) return LBQ_ERR_FORMAT;
    const Codebook& cbk = codebook();
    const int64_t ng = K / kGroup;
    parallel_for(N, [&](int64_t b, int64_t e) {
        for (int64_t n = b; n < e; ++n) {
            for (int64_t g = 0; g < ng; ++g) {
                const RecordAddr ra = record_addr(L, n, g);
                float* wrow = W_hat + n * K + g * kGroup;
                if (w4) {
                    uint16_t sh;
                    std::memcpy(&sh, in + ra.rec + kW4ScaleOff + uint64_t(ra.slot) * 2, 2);
                    const double s = f16_bits_to_f64(sh);
                    const uint8_t zb = in[ra.rec + kW4ZeroOff + (ra.slot >> 1)];
                    const double z = (g % 2 == 0) ? (zb & 15) : (zb >> 4);
                    const uint8_t* qb = in + ra.rec + uint64_t(ra.slot) * 16;
                    for (int k = 0; k < 16; ++k) {
                        const double lo = static_cast<double>(qb[k] & 15) - z, hi = static_cast<double>(qb[k] >> 4) - z;
                        wrow[k] = static_cast<float>(lo * s);
                        wrow[k + 16] = static_cast<float>(hi * s);
                    }
                } else {
                    uint16_t Sh, Zh;
                    std::memcpy(&Sh, in + ra.rec + kW2SOff + uint64_t(ra.slot) * 2, 2);
                    std::memcpy(&Zh, in + ra.rec + kW2ZOff + uint64_t(ra.slot) * 2, 2);
                    const double S = f16_bits_to_f64(Sh), Z = f16_bits_to_f64(Zh);
                    const uint8_t* cq = in + ra.rec + uint64_t(ra.slot) * 8;
                    for (int k = 0; k < kGroup; ++k) {
                        const double sc = S * cbk.val[(cq[k / 4] >> (2 * (k % 4))) & 3];
                        wrow[k] = static_cast<float>(sc + Z);
                    }
                }
            }
            // outlier columns: their exact FP16 values
            const uint64_t base = L.area_offset + uint64_t(n / lbq::kRowsPerBlock) * L.row_block_bytes +
                                  L.records * L.record_bytes;
            const int r = int(n % lbq::kRowsPerBlock);
            for (int32_t j = 0; j < n_out; ++j) {
                const int32_t rec = j / lbq::kOutlierCols;
                const uint64_t width = std::min<uint64_t>(
                    lbq::kOutlierCols, round_up(uint64_t(n_out), lbq::kOutlierColAlign) - uint64_t(rec) * lbq::kOutlierCols);
                uint16_t h;
                std::memcpy(&h, in + base + uint64_t(rec) * L.outlier_record_bytes +
                                    (uint64_t(r) * width + uint64_t(j % lbq::kOutlierCols)) * 2, 2);
                W_hat[n * K + idx[j]] = static_cast<float>(f16_bits_to_f64(h));
            }
        }
    });
    return LBQ_OK;
}

}  // extern "C"
