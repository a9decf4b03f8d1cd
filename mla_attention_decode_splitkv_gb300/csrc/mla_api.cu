// mla_api.cu -- C ABI of the MLA decode library: argument checks, the split-count
// heuristic, the per-device partial-result workspace, tensor-map encoding and launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "mla_decode.h"
#include "mla_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct Workspace {
  float* part_o = nullptr;
  float* part_lse = nullptr;
  int* status = nullptr;
  int* seq_count = nullptr;   // per-sequence piece counters, zero between calls
  long long slots = 0;
  long long counters = 0;
};

std::mutex g_mu;
Workspace g_ws[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_cc[kMaxDevices];
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_test_stall{0};
std::atomic<int> g_cross_rows{-1};

// Costs of the split model, in bytes (mla_decode_pick_splits; the header derives them).
constexpr double kPieceBytes = static_cast<double>(mla::kHeads) * (mla::kDimV + 1) * 4.0;  // 32,832
constexpr double kWaveBytes = 222e3;
constexpr double kCrossBytes = 300e3;
double row_bytes(int kv_dtype) {
  return kv_dtype == MLA_KV_BF16 ? 2.0 * mla::kDim
         : kv_dtype == MLA_KV_FP8_E4M3 ? 1.0 * mla::kDim
         : static_cast<double>(mla::kMxPacked + mla::kMxScales);
}
// A CTA's rate through the cache relative to the HBM rate: bf16 and fp8 CTAs stream at it; an
// MXFP4 CTA is bound by its dequantisation at 0.30 of it (2.02 of the 6.76 TB/s measured on
// GB300 at 256 x 8192).  The split model's costs (latencies and piece bytes at the HBM rate)
// count in the rows a CTA gets through in the same time: bytes x rate / row bytes.
double row_rate(int kv_dtype) { return kv_dtype == MLA_KV_MXFP4 ? 0.30 : 1.0; }
thread_local const char* t_last_cuda_error = "";

// Optional timing of each call's split kernel (events recorded on the call's stream).
struct ProfRecord {
  cudaEvent_t start, split_end, end;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;   // event pool, reused across begin/end cycles
size_t g_prof_n = 0;              // records used since begin

int note_cuda(cudaError_t e) {
  t_last_cuda_error = cudaGetErrorName(e);
  return MLA_ERR_CUDA;
}

// Device properties cached per device id (SM count, compute capability).
int device_info(int* dev_out, int* sms_out, int* cc_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return note_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  int sms = g_sm_count[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return note_cuda(e);
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return note_cuda(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return note_cuda(e);
    g_cc[dev].store(major * 10 + minor, std::memory_order_relaxed);
    g_sm_count[dev].store(sms, std::memory_order_release);   // published after the capability
  }
  *dev_out = dev;
  *sms_out = sms;
  *cc_out = g_cc[dev].load(std::memory_order_relaxed);
  return MLA_OK;
}

// Grow-only workspace of `slots` partial results and `counters` per-sequence counters on
// device `dev` (caller holds g_mu).  Counters are zeroed when allocated; the kernel leaves
// them at zero after every complete call.  A buffer is only replaced after a device-wide
// synchronisation, so no kernel still in flight (on any stream, enqueued by any thread)
// can use a freed buffer.
int ensure_workspace(int dev, long long slots, long long counters) {
  Workspace& w = g_ws[dev];
  if (w.status == nullptr) {
    cudaError_t e = cudaMalloc(&w.status, sizeof(int));
    if (e != cudaSuccess) { w.status = nullptr; cudaGetLastError(); return MLA_ERR_NO_MEMORY; }
    if ((e = cudaMemset(w.status, 0, sizeof(int))) != cudaSuccess) return note_cuda(e);
  }
  const bool grow_counters = counters > w.counters, grow_slots = slots > w.slots;
  if ((grow_counters && w.seq_count != nullptr) || (grow_slots && w.part_o != nullptr)) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return note_cuda(e);
  }
  if (grow_counters) {
    if (w.seq_count) { cudaFree(w.seq_count); w.seq_count = nullptr; }
    w.counters = 0;
    cudaError_t e = cudaMalloc(&w.seq_count, static_cast<size_t>(counters) * sizeof(int));
    if (e != cudaSuccess) { w.seq_count = nullptr; cudaGetLastError(); return MLA_ERR_NO_MEMORY; }
    if ((e = cudaMemset(w.seq_count, 0, static_cast<size_t>(counters) * sizeof(int))) != cudaSuccess) return note_cuda(e);
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return note_cuda(e);
    w.counters = counters;
  }
  if (!grow_slots) return MLA_OK;
  if (w.part_o) { cudaFree(w.part_o); w.part_o = nullptr; }
  if (w.part_lse) { cudaFree(w.part_lse); w.part_lse = nullptr; }
  w.slots = 0;
  const size_t o_bytes = static_cast<size_t>(slots) * mla::kHeads * mla::kDimV * sizeof(float);
  const size_t l_bytes = static_cast<size_t>(slots) * mla::kHeads * sizeof(float);
  if (cudaMalloc(&w.part_o, o_bytes) != cudaSuccess || cudaMalloc(&w.part_lse, l_bytes) != cudaSuccess) {
    cudaGetLastError();
    if (w.part_o) cudaFree(w.part_o);
    if (w.part_lse) cudaFree(w.part_lse);
    w.part_o = nullptr;
    w.part_lse = nullptr;
    return MLA_ERR_NO_MEMORY;
  }
  w.slots = slots;
  return MLA_OK;
}

long long slots_needed(int batch, int num_splits, int num_sms) {
  if (num_splits == 1) return 0;
  if (num_splits >= 2) return static_cast<long long>(batch) * num_splits;
  return static_cast<long long>(batch) + num_sms - 1;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace mla {

static int encode_map(CUtensorMap* map, const void* kv, int kv_dtype, bool rope, int box_rows = kBN) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return MLA_ERR_UNSUPPORTED;
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t rows = 1ull << 30;
  const bool bf = kv_dtype == MLA_KV_BF16, mx = kv_dtype == MLA_KV_MXFP4;
  const cuuint64_t width = mx ? kMxPacked : kDim;                       // elements per row
  cuuint64_t gdim[2] = {width, rows};
  cuuint64_t gstride[1] = {width * (bf ? 2 : 1)};                       // bytes per row
  cuuint32_t box[2] = {(bf || mx || rope) ? 64u : 128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                      const_cast<void*>(kv), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      (mx || rope) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

unsigned long long pipeline_wait_limit_ns() { return g_wait_limit_ns.load(); }

// The crossing's time (kCrossBytes is that time times one SM's HBM share) in the rows a CTA
// gets through in that time (row_rate).
int balance_cross_rows(int kv_dtype) {
  const int r = g_cross_rows.load();
  if (r >= 0) return r;
  return static_cast<int>(kCrossBytes / row_bytes(kv_dtype) * row_rate(kv_dtype) + 0.5);
}

int encode_kv_map(CUtensorMap* map, const void* kv, int kv_dtype) { return encode_map(map, kv, kv_dtype, false); }
int encode_rope_map(CUtensorMap* map, const void* kv) { return encode_map(map, kv, MLA_KV_FP8_E4M3, true); }
int encode_kv_map_rows(CUtensorMap* map, const void* kv, int kv_dtype, int box_rows) {
  return encode_map(map, kv, kv_dtype, false, box_rows);
}
int encode_rope_map_rows(CUtensorMap* map, const void* kv, int box_rows) {
  return encode_map(map, kv, MLA_KV_FP8_E4M3, true, box_rows);
}

}  // namespace mla

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_NO_MEMORY: return "MLA_ERR_NO_MEMORY";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    default: return "MLA_UNKNOWN_STATUS";
  }
}

const char* mla_last_cuda_error(void) { return t_last_cuda_error; }

void mla_decode_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : 1ull); }

void mla_decode_set_test_stall(int on) { g_test_stall = on ? 1 : 0; }

void mla_decode_set_cross_rows(int rows) { g_cross_rows = rows < 0 ? -1 : rows; }

int mla_decode_pick_splits(int batch, int kv_len_hint, int num_sms, int kv_dtype) {
  if (batch <= 0 || kv_len_hint < 0 || num_sms <= 0 || kv_dtype < 0 || kv_dtype > 2) return MLA_ERR_INVALID_ARG;
  // The split model of amd-mixed-mla submission 700955 (`_compute_custom_splits`: score =
  // utilisation of the CTA slots x L / (L + per-split overhead)), with this kernel's costs
  // written out in rows of the cache (one row = the bytes one cached token occupies):
  //  * a piece (partial output + log-sum-exp, 16 x 513 fp32) is written once, c rows, and
  //    read once by the CTA that merges its sequence, which reads all ns pieces in turn;
  //  * every wave of CTAs pays a CTA's start-up before its first copy and its drain after the
  //    last one: w rows, that latency (about 2 + 3 us, measured on GB300) times one SM's
  //    share of the HBM bandwidth (6.76 TB/s / 152 SMs);
  //  * in the balanced mode a CTA that moves from one sequence to the next drains and
  //    refills its pipeline (epilogue, piece count, q restaging): x rows, the crossing's
  //    measured latency (about 6.7 us) times the same share.
  // Time of the slowest CTA, in rows:
  //   uniform ns:  waves * (chunk + w + c [ns > 1]) + ns * c [ns > 1],
  //                waves = ceil(B ns / SMs), chunk = L / ns rounded up to 128-row tiles;
  //   balanced:    R + w + s c + (s - 1) x + p c,  R = B L / SMs rows per CTA, s = ceil(R / L) + 1
  //                sequences touched by a CTA, p = ceil(L / R) + 1 pieces per sequence.
  // The best uniform split count is returned, or 0 when the balanced mode is faster.
  // kv_dtype sets the row size and the CTAs' rate through the rows (row_rate), hence c, w and
  // x in rows.
  const double row = row_bytes(kv_dtype) / row_rate(kv_dtype);
  const double c = kPieceBytes / row, w = kWaveBytes / row, x = kCrossBytes / row;
  const long long L = std::max(kv_len_hint, 1), B = batch, S = num_sms, BN = mla::kBN;
  const long long ns_max = std::min<long long>(mla::kMaxSplits, (L + BN - 1) / BN);
  const double useful = static_cast<double>(B) * static_cast<double>(L) / static_cast<double>(S);
  int best_ns = 1;
  double best_t = 0.0;
  for (long long ns = 1; ns <= ns_max; ++ns) {
    const long long waves = (B * ns + S - 1) / S;
    const long long chunk = ((L + ns - 1) / ns + BN - 1) / BN * BN;
    const double t = waves * (chunk + w + (ns > 1 ? c : 0.0)) + (ns > 1 ? ns * c : 0.0);
    if (ns == 1 || t < best_t) { best_t = t; best_ns = static_cast<int>(ns); }
  }
  const double R = useful;
  const double s_seq = std::ceil(R / L) + 1.0, pieces = std::ceil(L / R) + 1.0;
  const double t_bal = R + w + s_seq * c + (s_seq - 1.0) * x + pieces * c;
  return t_bal < best_t ? 0 : best_ns;
}

int mla_decode_workspace_slots(int batch, int num_splits, int num_sms) {
  if (batch <= 0 || num_sms <= 0) return MLA_ERR_INVALID_ARG;
  long long s = slots_needed(batch, num_splits, num_sms);
  return s > 0x7fffffffLL ? MLA_ERR_INVALID_ARG : static_cast<int>(s);
}

int mla_decode_reserve_workspace(int slots) {
  if (slots < 0) return MLA_ERR_INVALID_ARG;
  int dev, sms, cc;
  int rc = device_info(&dev, &sms, &cc);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  return ensure_workspace(dev, slots, slots);
}

int mla_decode_release_workspace(void) {
  int dev, sms, cc;
  int rc = device_info(&dev, &sms, &cc);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[dev];
  cudaError_t e = cudaDeviceSynchronize();
  if (w.part_o) cudaFree(w.part_o);
  if (w.part_lse) cudaFree(w.part_lse);
  if (w.status) cudaFree(w.status);
  if (w.seq_count) cudaFree(w.seq_count);
  w = Workspace();
  return e == cudaSuccess ? MLA_OK : note_cuda(e);
}

int mla_decode_device_status(int clear) {
  int dev, sms, cc;
  int rc = device_info(&dev, &sms, &cc);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[dev];
  if (w.status == nullptr) return MLA_OK;
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, w.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return note_cuda(e);
  if (clear && v && (e = cudaMemset(w.status, 0, sizeof(int))) != cudaSuccess) return note_cuda(e);
  return (v & mla::kStatusTimeout) ? MLA_ERR_TIMEOUT : MLA_OK;
}

// Shared by mla_decode (page_size 0), mla_decode_paged and mla_decode_paged_multi
// (qo_indptr != null: `batch` counts query rows, `num_seqs` sequences).
static int decode_impl(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_indptr,
                       const int32_t* page_indices, const int32_t* last_page_len, int page_size,
                       const int32_t* qo_indptr, int num_seqs, void* out, int batch, int num_splits, int kv_dtype,
                       void* stream) {
  if (q == nullptr || kv == nullptr || kv_indptr == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  if (page_size != 0) {
    if (page_size < 1 || page_size > mla::kBN || (page_size & (page_size - 1)) != 0) return MLA_ERR_INVALID_ARG;
    if (page_indices == nullptr || last_page_len == nullptr) return MLA_ERR_INVALID_ARG;
    if (!aligned(page_indices, 4) || !aligned(last_page_len, 4)) return MLA_ERR_INVALID_ARG;
  }
  if (qo_indptr != nullptr && (page_size == 0 || num_seqs <= 0 || !aligned(qo_indptr, 4))) return MLA_ERR_INVALID_ARG;
  if (batch <= 0 || num_splits > mla::kMaxSplits) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_MXFP4) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_scale == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 8) || !aligned(kv_indptr, 4)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !aligned(kv_scale, 4)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_MXFP4 && !aligned(kv_scale, 2)) return MLA_ERR_INVALID_ARG;

  int dev, sms, cc;
  int rc = device_info(&dev, &sms, &cc);
  if (rc) return rc;
  if (cc != 103) return MLA_ERR_UNSUPPORTED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int ns = num_splits >= 1 ? num_splits : 0;
  // Several query tokens per sequence: bf16 and fp8 caches decode them two at a time (the
  // fused instances; the CTAs of odd-numbered tokens exit at once), MXFP4 one query row per CTA.
  const bool pairs = qo_indptr != nullptr && kv_dtype != MLA_KV_MXFP4;
  const int units = pairs ? (batch + 1) / 2 : batch;   // (an estimate: tokens per sequence may vary)
  if (qo_indptr != nullptr && ns == 0) ns = std::max(1, std::min(sms / units, mla::kMaxSplits));   // uniform only
  const long long grid_ll = ns >= 1 ? static_cast<long long>(batch) * ns : sms;
  if (grid_ll > 0x7fffffffLL) return MLA_ERR_INVALID_ARG;

  // The workspace lock is held until the launch is enqueued: a concurrent call (or a
  // reserve / release) on another host thread cannot replace these buffers in between.
  std::lock_guard<std::mutex> ws_lock(g_mu);
  rc = ensure_workspace(dev, slots_needed(batch, ns, sms), ns == 1 ? 0 : batch);
  if (rc) return rc;
  const Workspace ws = g_ws[dev];

  mla::DecodeParams p;
  // Tiled boxes of one page (8+ rows), of one row for the four-row gathers of smaller pages,
  // of 128 rows for a contiguous cache.
  const int box_rows = page_size >= mla::kMinPage ? page_size : (page_size > 0 ? 1 : mla::kBN);
  rc = mla::encode_kv_map_rows(&p.tmap, kv, kv_dtype, box_rows);
  if (rc) return rc;
  if (kv_dtype == MLA_KV_FP8_E4M3) {
    rc = mla::encode_rope_map_rows(&p.tmap_rope, kv, box_rows);
    if (rc) return rc;
  }
  p.page_size = page_size;
  p.page_shift = 0;
  while ((1 << p.page_shift) < page_size) ++p.page_shift;
  p.page_indices = page_indices;
  p.last_page_len = last_page_len;
  p.qo_indptr = qo_indptr;
  p.num_seqs = num_seqs;
  p.pair_rows = pairs ? 1 : 0;
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint8_t*>(kv);
  p.kv_scale = kv_scale;
  p.kv_indptr = kv_indptr;
  p.out = static_cast<uint16_t*>(out);
  p.part_o = ws.part_o;
  p.part_lse = ws.part_lse;
  p.status = ws.status;
  p.seq_count = ws.seq_count;
  p.batch = batch;
  p.num_splits = ns;
  p.num_ctas = static_cast<int>(grid_ll);
  p.logit_scale_log2 = static_cast<float>((1.0 / std::sqrt(static_cast<double>(mla::kDim))) * 1.4426950408889634);
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.test_stall = g_test_stall.load();
  p.cross_rows = mla::balance_cross_rows(kv_dtype);

  ProfRecord rec{nullptr, nullptr, nullptr};
  bool prof = false;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) {
      if (g_prof_n == g_prof.size()) {
        ProfRecord r{nullptr, nullptr, nullptr};
        cudaEventCreate(&r.start);
        cudaEventCreate(&r.split_end);
        cudaEventCreate(&r.end);
        g_prof.push_back(r);
      }
      rec = g_prof[g_prof_n++];
      prof = true;
    }
  }
  if (prof) cudaEventRecord(rec.start, st);
  cudaError_t e = page_size != 0 ? mla::launch_split_paged(kv_dtype, p, static_cast<int>(grid_ll), st)
                                  : mla::launch_split(kv_dtype, p, static_cast<int>(grid_ll), st);
  if (e != cudaSuccess) return note_cuda(e);
  if (prof) {
    cudaEventRecord(rec.split_end, st);
    cudaEventRecord(rec.end, st);
  }
  return MLA_OK;
}

int mla_decode(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_indptr, void* out, int batch,
               int num_splits, int kv_dtype, void* stream) {
  return decode_impl(q, kv, kv_scale, kv_indptr, nullptr, nullptr, 0, nullptr, 0, out, batch, num_splits, kv_dtype,
                     stream);
}

int mla_decode_paged(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_page_indptr,
                     const int32_t* kv_page_indices, const int32_t* kv_last_page_len, int page_size, void* out,
                     int batch, int num_splits, int kv_dtype, void* stream) {
  if (page_size == 0) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv, kv_scale, kv_page_indptr, kv_page_indices, kv_last_page_len, page_size, nullptr, 0, out,
                     batch, num_splits, kv_dtype, stream);
}

int mla_decode_paged_multi(const void* q, const int32_t* qo_indptr, int total_q, const void* kv, const void* kv_scale,
                           const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                           const int32_t* kv_last_page_len, int page_size, void* out, int batch, int num_splits,
                           int kv_dtype, void* stream) {
  if (page_size == 0 || qo_indptr == nullptr || total_q <= 0 || batch <= 0) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv, kv_scale, kv_page_indptr, kv_page_indices, kv_last_page_len, page_size, qo_indptr, batch,
                     out, total_q, num_splits, kv_dtype, stream);
}

int mla_decode_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_n = 0;
  g_prof_on = true;
  return MLA_OK;
}

int mla_decode_profile_end(double* split_ms, double* call_ms, int* calls) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  double s = 0.0, t = 0.0;
  int n = 0;
  int rc = MLA_OK;
  for (size_t i = 0; i < g_prof_n; ++i) {
    const ProfRecord& r = g_prof[i];
    float a = 0.f, b = 0.f;
    cudaError_t e1 = cudaEventSynchronize(r.end);
    cudaError_t e2 = cudaEventElapsedTime(&a, r.start, r.split_end);
    cudaError_t e3 = cudaEventElapsedTime(&b, r.start, r.end);
    if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
      rc = note_cuda(e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
    } else {
      s += a;
      t += b;
      ++n;
    }
  }
  g_prof_n = 0;
  if (split_ms) *split_ms = s;
  if (call_ms) *call_ms = t;
  if (calls) *calls = n;
  return rc;
}

}  // extern "C"
