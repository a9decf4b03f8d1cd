// mla_internal.h -- parameters shared by the host launcher and the device kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mla {

constexpr int kHeads = 16;
constexpr int kDim = 576;
constexpr int kDimV = 512;
constexpr int kBN = 128;           // cached tokens per tile (= UMMA M)
constexpr int kMinPage = 8;        // smallest page (rows) a TMA box loads whole: one swizzle atom; 1-4: see run_producer_sp
constexpr int kMxBlock = 32;
constexpr int kMxPacked = 288;     // bytes of e2m1 nibbles per row
constexpr int kMxScales = 18;      // e8m0 scales per row
constexpr int kMaxSplits = 4096;
constexpr int kBalancedMinTokens = 256;  // fewest tokens a persistent CTA is given

// Status bits of the device status word.
constexpr int kStatusTimeout = 1;

struct DecodeParams {
  CUtensorMap tmap;                // KV rows as a 2D tensor (see encode_kv_map)
  CUtensorMap tmap_rope;           // fp8: the rope bytes [512, 576) of each row, 64-byte boxes
  const uint16_t* q;               // bf16 bits [batch][16][576]
  const uint8_t* kv;               // raw cache base
  const void* kv_scale;            // fp8: const float*; mxfp4: const uint8_t* [T][18]
  const int32_t* kv_indptr;        // [batch + 1]
  uint16_t* out;                   // bf16 bits [batch][16][512]
  float* part_o;                   // [slots][16][512] normalised partial outputs
  float* part_lse;                 // [slots][16]      log2-domain log-sum-exp of the partials
  int* status;                     // device status word
  int* seq_count;                  // [batch] pieces written per sequence (zero between calls)
  int batch;
  int num_splits;                  // >= 1: uniform splits per sequence; 0: balanced over CTAs
  int num_ctas;                    // grid size (balanced mode: persistent CTAs)
  float logit_scale_log2;          // sm_scale * log2(e)
  unsigned long long wait_limit_ns;
  int test_stall;                  // test hook: the QK issuer waits on a barrier that never completes
  // Paged cache (mla_decode_paged; 0 / null otherwise): kv_indptr indexes page_indices.
  int page_size;                   // rows per page: a power of two, 1 .. 128
  int page_shift;                  // log2(page_size)
  const int32_t* page_indices;     // [kv_indptr[batch]] physical page of each sequence page
  const int32_t* last_page_len;    // [sequences] rows used in each sequence's last page (1..page_size)
  // Several query tokens per sequence (mla_decode_paged_multi; null otherwise, uniform splits
  // only): batch counts query rows, qo_indptr [num_seqs + 1] maps sequences to query rows.
  const int32_t* qo_indptr;
  int num_seqs;
  int pair_rows;                   // fused multi-token instances: a CTA decodes query rows t, t + 1 together
  // Balanced mode, contiguous cache: the cost in rows of each sequence start after the first
  // (see balanced_cost_total in the kernel; 0 cuts by rows alone).
  int cross_rows;
};


// Tensor map of the cache rows for the kernel's TMA loads.  bf16: [rows x 576] bf16,
// 64-element boxes, 128-byte swizzle; fp8: [rows x 576] bytes, 128-byte boxes, 128-byte
// swizzle; MXFP4: the packed nibbles [rows x 288] bytes, 64-byte boxes, 64-byte swizzle.
// All boxes are 128 rows.  The row count is an upper bound: the kernel never addresses a
// row at or past kv_indptr[batch] (its 128-row windows end at the last row of a sequence;
// rows before row 0 are zero-filled by the TMA).  Returns an MLA_* status.
int encode_kv_map(CUtensorMap* map, const void* kv, int kv_dtype);
// fp8 caches: the same rows with 64-byte boxes and 64-byte swizzle (the rope chunk).
int encode_rope_map(CUtensorMap* map, const void* kv);

// The pipeline wait limit set by mla_decode_set_wait_limit_ns (default 2 s).
unsigned long long pipeline_wait_limit_ns();

// DecodeParams::cross_rows for a cache dtype: the split model's crossing cost in rows of that
// cache (or the value set by mla_decode_set_cross_rows).
int balance_cross_rows(int kv_dtype);

// Launches the split kernel for kv_dtype (geometry per dtype is internal to mla_split.cu).
cudaError_t launch_split(int kv_dtype, const DecodeParams& p, int grid, cudaStream_t stream);
// The same for a paged cache (page size 1 .. 128, a power of two; TMA boxes of page_size rows
// from 8 rows up; four-row gathers (bf16, fp8) or 16-byte cp.async copies (MXFP4) below).
cudaError_t launch_split_paged(int kv_dtype, const DecodeParams& p, int grid, cudaStream_t stream);
// Tensor maps with boxes of `box_rows` rows (paged caches: box_rows = page size).
int encode_kv_map_rows(CUtensorMap* map, const void* kv, int kv_dtype, int box_rows);
int encode_rope_map_rows(CUtensorMap* map, const void* kv, int box_rows);

}  // namespace mla
