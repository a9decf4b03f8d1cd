// mla_noalloc.cu -- mla_decode_noalloc: the same decode as mla_decode, for callers that
// must not allocate device memory.
//
// Some callers cannot call cudaMalloc on the decode path: a serving engine or plugin host
// that owns every device allocation through its own pre-sized pool and forbids stray ones,
// or a latency-critical loop that cannot afford cudaMalloc/cudaFree (cudaFree synchronises
// the whole device).  mla_decode grows a library-owned workspace with cudaMalloc on first
// use; this entry point instead keeps its scratch (the split partial results, the
// per-sequence piece counters and the kernel status word) in a fixed-size array that lives
// in the library's device module.
//
// The array is a file-scope static __device__ object, so every GPU that loads this library
// holds kNoallocScratchBytes of it until the process exits.  Host code cannot use the
// array's name as a device address: on the first call on each device (with that device
// current) the address is looked up once with cudaGetSymbolAddress and cached.  That first
// call therefore does one-time set-up work and should happen before any stream capture.
// All calls share the one array and it keeps the previous call's contents, so calls that
// overlap on the GPU (different streams, no ordering between them) race on it.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_decode.h"
#include "mla_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kSlotBytes = static_cast<size_t>(mla::kHeads) * mla::kDimV * sizeof(float);   // partial O
constexpr size_t kLseBytes = static_cast<size_t>(mla::kHeads) * sizeof(float);                 // partial lse
constexpr size_t kStatusBytes = 256;
constexpr size_t kCounterBytes = static_cast<size_t>(MLA_NOALLOC_MAX_SLOTS) * sizeof(int);
constexpr size_t kNoallocScratchBytes =
    static_cast<size_t>(MLA_NOALLOC_MAX_SLOTS) * (kSlotBytes + kLseBytes) + kStatusBytes + kCounterBytes;

// Layout: [status word (256 B)] [piece counters: slots x int32] [partial O: slots x 16 x 512 fp32]
//         [partial lse: slots x 16 fp32]
// The status word and the counters are contiguous so that one stream-ordered memset per
// call re-arms both (a call that splits sequences uses counters [0, batch), and a call
// needing partial slots has batch <= slots, so the counters always fit).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr size_t kCountersOffset = kStatusBytes;
constexpr size_t kPartOOffset = kStatusBytes + kCounterBytes;
constexpr size_t kPartLseOffset = kPartOOffset + static_cast<size_t>(MLA_NOALLOC_MAX_SLOTS) * kSlotBytes;
static_assert(kPartOOffset % 256 == 0, "partial outputs must stay 16-byte aligned");

std::mutex g_mu;
void* g_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device,
// with that device current); nullptr on failure.
unsigned char* scratch_base(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_addr[dev] = ptr;
  }
  return static_cast<unsigned char*>(g_addr[dev]);
}
}  // namespace

extern "C" int mla_decode_noalloc(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_indptr,
                                  void* out, int batch, int num_splits, int kv_dtype, void* stream) {
  if (q == nullptr || kv == nullptr || kv_indptr == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  if (batch <= 0 || num_splits > mla::kMaxSplits) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_MXFP4) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_scale == nullptr) return MLA_ERR_INVALID_ARG;
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 8) || !aligned(kv_indptr, 4)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !aligned(kv_scale, 4)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_MXFP4 && !aligned(kv_scale, 2)) return MLA_ERR_INVALID_ARG;

  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (major * 10 + minor != 103) return MLA_ERR_UNSUPPORTED;

  const int ns = num_splits >= 1 ? num_splits : 0;
  const long long grid = ns >= 1 ? static_cast<long long>(batch) * ns : sms;
  const long long slots = ns == 1 ? 0 : (ns >= 2 ? static_cast<long long>(batch) * ns : static_cast<long long>(batch) + sms - 1);
  if (slots > MLA_NOALLOC_MAX_SLOTS || grid > 0x7fffffffLL) return MLA_ERR_NO_MEMORY;  // beyond the fixed scratch

  unsigned char* b = scratch_base(dev);
  if (b == nullptr) return MLA_ERR_CUDA;
  int* status = reinterpret_cast<int*>(b);
  int* seq_count = reinterpret_cast<int*>(b + kCountersOffset);
  float* part_o = reinterpret_cast<float*>(b + kPartOOffset);
  float* part_lse = reinterpret_cast<float*>(b + kPartLseOffset);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Each call starts from a zero status word and zero piece counters: one stream-ordered
  // memset over both (the kernels only ever set status bits, and a call cut short by a
  // pipeline timeout may leave its counters mid-count).
  const size_t clear_bytes = kStatusBytes + (ns == 1 ? 0 : static_cast<size_t>(batch) * sizeof(int));
  if (cudaMemsetAsync(status, 0, clear_bytes, st) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }

  mla::DecodeParams p;
  int rc = mla::encode_kv_map(&p.tmap, kv, kv_dtype);
  if (rc) return rc;
  if (kv_dtype == MLA_KV_FP8_E4M3 && (rc = mla::encode_rope_map(&p.tmap_rope, kv)) != 0) return rc;
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint8_t*>(kv);
  p.kv_scale = kv_scale;
  p.kv_indptr = kv_indptr;
  p.out = static_cast<uint16_t*>(out);
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.status = status;
  p.seq_count = seq_count;
  p.batch = batch;
  p.num_splits = ns;
  p.num_ctas = static_cast<int>(grid);
  p.logit_scale_log2 = static_cast<float>((1.0 / std::sqrt(static_cast<double>(mla::kDim))) * 1.4426950408889634);
  p.wait_limit_ns = mla::pipeline_wait_limit_ns();
  p.test_stall = 0;
  p.page_size = 0;
  p.page_shift = 0;
  p.page_indices = nullptr;
  p.last_page_len = nullptr;
  p.qo_indptr = nullptr;
  p.num_seqs = 0;
  p.pair_rows = 0;
  p.cross_rows = mla::balance_cross_rows(kv_dtype);
  if (mla::launch_split(kv_dtype, p, static_cast<int>(grid), st) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return MLA_OK;
}

extern "C" int mla_decode_noalloc_status(int clear) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) { cudaGetLastError(); return MLA_ERR_CUDA; }
  unsigned char* b = scratch_base(dev);
  if (b == nullptr) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, b, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }
  if (clear && v && cudaMemset(b, 0, sizeof(int)) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return (v & mla::kStatusTimeout) ? MLA_ERR_TIMEOUT : MLA_OK;
}
