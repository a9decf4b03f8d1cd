// mla_split.cu -- the split-KV flash-decode kernel (tcgen05 / TMA, sm_103a) for
// single-token MLA decode, with the log-sum-exp merge of the splits fused in.
//
// Method (amd-mixed-mla submissions 727205 `mla_s1`/`mla_rd`, 700955 `mla_attn_v71`/
// `reduce_lse_v71`, 599694 `_flash_fp8_split_s1`/`_s2`): every (sequence, split) pair
// runs an online softmax over its cached rows and emits a normalised partial output plus
// its log-sum-exp; the partials are merged by log-sum-exp weights.  Here the CTA that
// writes a sequence's last partial merges them (per-sequence counters), so one call is one
// launch.  The GB300 design:
//
//  * "swap-AB" tensor-core formulation, so the 16 heads sit on the MMA's N side:
//        S^T[128 tok x 16 h]   = K_tile[128 x 576] . Q^T          (UMMA M = 128 tokens)
//        O^T[512 dim x 16 h]  += V_tile^T[512 x 128] . P^T        (4 UMMAs of M = 128 dims)
//    K_tile and V_tile are the same shared-memory bytes (V = first 512 columns of a
//    cached row): K-major for QK^T, MN-major for PV.  Accumulators live in TMEM.
//  * fp8 caches feed the e4m3 tensor cores directly (kind::f8f6f4, no dequantisation);
//    q and P are carried exactly-enough as two e4m3 terms (hi + lo/16) stacked on N, so
//    N = 32 and the contraction error stays at the bf16 level.  The per-tensor kv_scale
//    is folded into the logit multiplier and the final output.
//  * bf16 caches use kind::f16 with bf16 q and P (N = 16).
//  * MXFP4 caches are dequantised in shared memory by four extra warps into an e4m3
//    "carrier" (per-block shift tables, per-row power-of-two factor applied by the softmax)
//    and then take the fp8 path.
//  * KV rows stream HBM -> SMEM with 2D TMA through an mbarrier ring that one producer
//    warp fills; one warp issues the QK^T MMAs and two warps the PV MMAs; eight warps run
//    the online softmax (one token per thread = one TMEM lane, eight heads each), the rare
//    lazy O rescale in TMEM, the epilogue and the merge.
//  * Online softmax in the log2 domain with a lazy reference maximum: O is rescaled only
//    when a tile's maximum exceeds the reference by more than kTau (log2 units).
//
// Every pipeline wait is bounded: on timeout the kernel sets the device status word and
// all roles leave their loops; in-flight copies and MMAs are drained (bounded) before the
// tensor memory is released.
#include <cstddef>
#include <mutex>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
using namespace ptx;

namespace {

constexpr float kNegInf = -__builtin_huge_valf();
// Waits for a CTA's own copies and MMAs in flight (before it exits, also after a give-up)
// keep this limit whatever the pipeline wait limit is, so that no CTA ends with an async
// write to its shared memory or an MMA still reading it.
constexpr unsigned long long kDrainLimitNs = 2000000000ull;

// ---------------------------------------------------------------- per-dtype geometry
template <int KV>
struct Cfg;
template <>
struct Cfg<0> {                    // bf16 cache
  static constexpr int kSlotBytes = 32768;   // two [128 x 64 bf16] SW128 boxes
  static constexpr int kRing = 6;
  static constexpr int kSPT = 5;             // chunks per tile: 4 x 128 value dims + rope
  static constexpr int kRingPT = 5;          // ring slots per tile (the rope chunk rides in the ring)
  static constexpr int kRopeSlots = 0;
  static constexpr int kN = 16;
  static constexpr int kQBytes = 9 * 2048;   // 9 chunks of [16 rows x 128 B]
  static constexpr int kTmemCols = 128;
  static constexpr int kSCols = 16;
  static constexpr int kOCols = 16;
  static constexpr float kTau = 8.0f;
  static constexpr int kSoftWarps = 8;
  static constexpr int kDeqWarps = 0;
  static constexpr int kThreads = 384;       // producer, QK issuer, 2 PV issuers, 8 softmax warps
};
template <>
struct Cfg<1> {                    // fp8 e4m3 cache
  static constexpr int kSlotBytes = 16384;   // one [128 x 128 B] SW128 box
  static constexpr int kRing = 11;           // value chunks only (2.75 tiles)
  static constexpr int kSPT = 5;
  static constexpr int kRingPT = 4;
  static constexpr int kRopeSlots = 2;       // rope chunks: [128 x 64 B] SW64 slots of their own
  static constexpr int kN = 32;              // 16 hi heads + 16 lo heads
  static constexpr int kQBytes = 4 * 4096 + 2048;   // 4 chunks of [32 rows x 128 B] SW128 + rope [32 x 64 B] SW64
  static constexpr int kTmemCols = 256;
  static constexpr int kSCols = 32;
  static constexpr int kOCols = 32;
  static constexpr float kTau = 4.0f;        // P <= 16 -> 16 P <= 256 fits e4m3
  static constexpr int kSoftWarps = 8;
  static constexpr int kDeqWarps = 0;
  static constexpr int kThreads = 384;       // producer, QK issuer, 2 PV issuers, 8 softmax warps
};

template <>
struct Cfg<2> {                    // MXFP4 cache: dequantised to an e4m3 carrier in SMEM
  static constexpr int kSlotBytes = 16384;
  static constexpr int kRing = 8;            // value chunks of exactly two tiles
  static constexpr int kSPT = 5;
  static constexpr int kRingPT = 4;          // the rope chunk has its own [128 x 64 B] SW64 buffer
  static constexpr int kRopeSlots = 2;       // rope carrier, double-buffered
  static constexpr int kN = 32;
  static constexpr int kQBytes = 4 * 4096 + 2048;
  static constexpr int kTmemCols = 256;
  static constexpr int kSCols = 32;
  static constexpr int kOCols = 32;
  static constexpr float kTau = 4.0f;
  static constexpr int kSoftWarps = 8;
  static constexpr int kRowThreads = 1;      // dequant threads per carrier row
  static constexpr int kDeqWarps = 4 * kRowThreads;
  static constexpr int kThreads = 32 * (4 + kSoftWarps + kDeqWarps);   // issuers, softmax, dequant
  // Registers per thread after the role split (launch: 128 each): the issuer and dequant
  // warpgroups give registers up to the softmax warpgroups.
  // 32 * (4 * 72 + 8 * 160 + 4 * 120) = 65536 = 512 * 128.  (The dequantisation loop gains
  // from the larger budget: 256 x 8192 at 80 / 168 / 96 took 327 us, at 72 / 160 / 120 318.)
  static constexpr int kRegsIssue = 72;
  static constexpr int kRegsSoft = 160;
  static constexpr int kRegsDeq = 120;
  static constexpr int kRegsNeeded = 32 * (4 * kRegsIssue + kSoftWarps * kRegsSoft + kDeqWarps * kRegsDeq);
};
static_assert(Cfg<2>::kRegsNeeded <= 65536, "MXFP4 register split exceeds the register file");

constexpr int kPBytes = 4096;      // one P^T buffer: [128 tokens x 32 B] SW32 (one query token)
constexpr int kSlabBytes = 8192;   // MXFP4 staging: 64 packed bytes (4 blocks) of each of 128 rows, SW64
constexpr int kSlabs = 5;          // slab ring: a tile is 5 slabs (4 value chunks + rope)
// MXFP4 tiles are fetched, converted and multiplied rope chunk first: its carrier buffer is
// freed by the QK MMAs of the previous tile, so the dequantisation of tile g can start on it
// while the PV MMAs of tile g - 2 still read the value slots it needs next.
// Chunk i of an MXFP4 tile in fetch / conversion / QK order (4 = the rope chunk).
__host__ __device__ constexpr int mx_chunk(int i) { return i == 0 ? 4 : i - 1; }
constexpr int kLutCount = 14;      // e2m1 -> e4m3 tables for block shifts 0..-12, then zero
// Smallest MXFP4 row exponent e_i (biased): blocks more than 12 binades below it decode to
// zero, so a row whose largest block is below 2^-64 (|value| < 6 * 2^-64) reads as zeros.
constexpr int kRowExpFloor = 127 - 64;
constexpr int kRopeBytes = 8192;   // one rope slot: [128 rows x 64 B] SW64 (fp8 cache bytes / MXFP4 carrier)

struct SharedState {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t q_ready;
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t o_free;
  uint64_t mma_done[3];
  uint64_t never;                  // test hook: a barrier nothing arrives on
  alignas(16) float red[2][4][32];  // read as float4; [token * 16 + head]
  alignas(16) float lsum[4][32];
  alignas(16) float qscale[32];
  uint64_t slab_full[kSlabs];      // MXFP4 only
  uint64_t slab_empty[kSlabs];
  uint64_t etok_full[4];
  uint64_t rope_full[2];           // rope slots (fp8: TMA, MXFP4: dequant) / consumed by QK
  uint64_t rope_empty[2];
  int etok[4][128];                // per-row max block exponent of the last 4 tiles
  int sp_rows[128];                // MXFP4, pages of 1-4 rows: the cache row of each window row of a tile
  uint2 lut[kLutCount];            // 8 e4m3 bytes per block shift
  long long seg_total;              // kv_indptr[batch] (balanced mode)
  long long seg_lo, seg_hi;        // this CTA's position range (balanced mode)
  int seg_b0;                      // first sequence of this CTA (balanced mode)
  int merge_slot0;                 // fused merge: first slot and piece count to merge
  int merge_pieces;
  uint32_t tmem_base;
  int abort;
};

static_assert(offsetof(SharedState, red) % 16 == 0, "float4 reads of SharedState::red need 16-byte alignment");
static_assert(offsetof(SharedState, lut) % 8 == 0, "uint2 reads of SharedState::lut need 8-byte alignment");

// Geometry of a kernel instance that decodes QL query tokens of a sequence at once (QL = 2:
// the fused multi-token instances).  The QL x 16 query rows (x 2 e4m3 terms for fp8) sit on
// the MMAs' N side, so each cached tile is read once for all of them.  QL = 1 is Cfg<KV> as is.
template <int KV, int QL>
struct Geo {
  using C = Cfg<KV>;
  static_assert(QL == 1 || (QL == 2 && KV != 2), "fused multi-token instances: bf16 and fp8 caches");
  static constexpr int kN = C::kN * QL;                 // MMA N: query rows (x2 for the e4m3 hi + lo terms)
  static constexpr int kSCols = C::kSCols * QL;         // TMEM columns of one S buffer
  static constexpr int kOCols = C::kOCols * QL;         // TMEM columns of one O block (128 dims)
  static constexpr int kTokCols = C::kSCols;            // columns per query token (in S and in O)
  static constexpr int kTmemCols = QL == 1 ? C::kTmemCols : (2 * kSCols + 4 * kOCols <= 256 ? 256 : 512);
  static constexpr int kQBytes = C::kQBytes * QL;
  static constexpr int kQChunk = (KV == 0 ? 2048 : 4096) * QL;   // one K-major q chunk [rows x 128 B]
  static constexpr int kPBuf = kPBytes * QL;            // one P^T buffer: [128 tokens x 32 QL B]
  // P^T buffers: two (tile parity), or one in the fused two-token fp8 instance, whose softmax
  // writes P of tile g after the PV MMAs of tile g - 1 have read theirs (they complete well
  // before the softmax of tile g gets that far), so that its ring keeps a tenth slot.
  static constexpr int kPBufs = (QL == 2 && KV == 1) ? 1 : 2;
  // The second query token's q (and P^T) take ring slots: fp8 keeps 10 (2.5 tiles), bf16 one
  // tile's 5.
  static constexpr int kRing = QL == 1 ? C::kRing : (KV == 1 ? 10 : C::kRingPT);
  // Register split (setmaxnreg) after the role dispatch: MXFP4 (issuers / softmax / dequant)
  // and the fused two-token fp8 instance, whose softmax holds both tokens' hi and lo columns
  // (issuers / softmax: 128 * 88 + 256 * 208 = 64512 = 384 * 168).
  static constexpr bool kSplitRegs = KV == 2 || (KV == 1 && QL == 2);
  static constexpr int kRegsIssue = KV == 2 ? Cfg<2>::kRegsIssue : 88;
  static constexpr int kRegsSoft = KV == 2 ? Cfg<2>::kRegsSoft : 208;
  static constexpr int kRegsNeeded = KV == 2 ? Cfg<2>::kRegsNeeded : 32 * (4 * kRegsIssue + C::kSoftWarps * kRegsSoft);
};

template <int KV>
__host__ __device__ constexpr size_t raw_bytes() {
  return KV == 2 ? (size_t)kSlabs * kSlabBytes : 0;
}
template <int KV>
__host__ __device__ constexpr size_t rope_bytes() {
  return (size_t)Cfg<KV>::kRopeSlots * kRopeBytes;
}
template <int KV, int QL = 1>
__host__ __device__ constexpr size_t smem_bytes() {
  using G = Geo<KV, QL>;
  return 1024 + (size_t)G::kRing * Cfg<KV>::kSlotBytes + rope_bytes<KV>() + G::kQBytes + G::kPBufs * G::kPBuf +
         raw_bytes<KV>() + sizeof(SharedState);
}
static_assert(smem_bytes<2>() <= 232448, "MXFP4 shared memory exceeds 227 KB");
static_assert(smem_bytes<1>() <= 232448, "fp8 shared memory exceeds 227 KB");
static_assert(smem_bytes<0>() <= 232448, "bf16 shared memory exceeds 227 KB");
static_assert(smem_bytes<1, 2>() <= 232448, "fused two-token fp8 shared memory exceeds 227 KB");
static_assert(smem_bytes<0, 2>() <= 232448, "fused two-token bf16 shared memory exceeds 227 KB");

// ---------------------------------------------------------------- work decomposition
struct Seg {
  int rows;    // query rows decoded together: 1, or 2 in the fused multi-token instances
  int b;       // batch row (the first of the `rows` query rows)
  int row0;    // kv_indptr[b] (paged: the sequence's first entry in the page list)
  int n_total; // tokens in the sequence
  int n_lo;    // token range [n_lo, n_hi) within the sequence
  int n_hi;
  int slot;    // partial-result slot (when !direct)
  bool direct; // the range is the whole sequence: write the bf16 output directly
};

__device__ __forceinline__ int balanced_ctas(long long total, int G) {
  long long need = (total + kBalancedMinTokens - 1) / kBalancedMinTokens;
  if (need < 1) need = 1;
  return static_cast<int>(need < G ? need : G);
}
// Paged cache: positions are rows of the page space (page-list entry i covers positions
// [i P, (i + 1) P)), and the cut points are rounded down to multiples of 128 so that every
// tile starts on a page boundary.  Consecutive cut points stay more than 128 apart (each
// CTA is given at least 256 positions before rounding), so no range is empty.
template <bool PG>
__device__ __forceinline__ long long cta_lo(int c, long long total, int Ge) {
  if constexpr (PG) {
    if (c >= Ge) return total;
    return static_cast<long long>(c) * total / Ge / kBN * kBN;
  }
  return static_cast<long long>(c) * total / Ge;
}
// Largest CTA index whose range starts at or before token x.
template <bool PG>
__device__ __forceinline__ int cta_of_token(long long x, long long total, int Ge) {
  int lo = 0, hi = Ge - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cta_lo<PG>(mid, total, Ge) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// First b in [0, batch) with kv_indptr[b + 1] > lo (batch if none); called by a full warp.
// Each round probes 32 evenly spaced entries at once, so a batch of B sequences costs
// ceil(log32(B)) dependent loads instead of log2(B).
__device__ int warp_first_seq(const int32_t* ip, int batch, long long lo) {
  const int lane = threadIdx.x & 31;
  int base = 0, count = batch;
  while (count > 32) {
    const int step = (count + 31) / 32;
    const int bi = base + min(count - 1, lane * step + step - 1);
    const bool f = lane * step < count && ip[bi + 1] > lo;
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (m == 0) return base + count;
    const int c = __ffs(m) - 1;
    base += c * step;
    count = min(step, count - c * step);
  }
  const bool f = lane < count && ip[base + lane + 1] > lo;
  const unsigned m = __ballot_sync(0xffffffffu, f);
  return m ? base + __ffs(m) - 1 : base + count;
}

// Contiguous cache, balanced mode: the CTAs share the batch's cost, not its rows.  Every
// sequence start after the first costs X rows more (X = cross_rows: the time a CTA loses
// when it moves from one sequence to the next, as the split model states it), so position
// r of sequence b sits at cost r + X b and the batch costs Tc = total + X (batch - 1).  CTA
// c owns costs [c Tc / Ge, (c + 1) Tc / Ge); a cost inside sequence b maps back to the
// position cost - X b, a cost in the X-gap before sequence b + 1 to that sequence's first
// position.  The map is monotone, so ranges stay contiguous and ordered; a range that lies
// inside one gap is empty (its CTA has no work).
__device__ __forceinline__ long long balanced_cost_total(long long total, int batch, long long X) {
  return total + X * (batch - 1);
}
// Largest CTA c < Ge with c Tc / Ge <= cost (the CTA that owns a position of that cost).
__device__ __forceinline__ int cta_of_cost(long long cost, long long Tc, int Ge) {
  const long long c = ((cost + 1) * Ge - 1) / Tc;
  return static_cast<int>(c < Ge - 1 ? c : Ge - 1);
}
// For two costs at once: the first b in [0, batch) with kv_indptr[b + 1] + X (b + 1) > C,
// i.e. the sequence whose cost range (with the gap after it) holds C (batch if none).
// Called by a full warp; each round probes 32 evenly spaced entries per cost, and the two
// searches' loads are issued together.
__device__ void warp_first_seq_cost2(const int32_t* ip, int batch, long long X, long long C0, long long C1,
                                     int* out0, int* out1) {
  const int lane = threadIdx.x & 31;
  const long long C[2] = {C0, C1};
  int base[2] = {0, 0}, count[2] = {batch, batch}, res[2] = {batch, batch};
  bool fin[2] = {false, false};
  while (!(fin[0] && fin[1])) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (fin[k]) continue;
      const int step = count[k] > 32 ? (count[k] + 31) / 32 : 1;
      const int bi = base[k] + min(count[k] - 1, lane * step + step - 1);
      const bool f = lane * step < count[k] && static_cast<long long>(ip[bi + 1]) + X * (bi + 1) > C[k];
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (m == 0) { res[k] = base[k] + count[k]; fin[k] = true; continue; }
      const int c = __ffs(m) - 1;
      if (step == 1) { res[k] = base[k] + c; fin[k] = true; continue; }
      base[k] += c * step;
      count[k] = min(step, count[k] - c * step);
    }
  }
  *out0 = res[0];
  *out1 = res[1];
}

// Enumerates the (sequence, token range) segments one CTA works on.
//  uniform (num_splits >= 1): CTA = b * ns + s, one segment (possibly empty), chunk rule
//     chunk = ceil(ceil(L/ns)/BN)*BN (amd-mixed-mla submission 727205, `mla_s1`).
//  balanced (num_splits == 0): CTA c owns tokens [c*T/G, (c+1)*T/G) of the concatenated
//     batch (T = kv_indptr[batch]); each sequence it touches is one non-empty segment;
//     partial slot = b + c (unique: the (b, c) pairs form a monotone staircase).
template <bool PG>
struct SegIter {
  long long lo, hi;
  int b, split, ns, cta;
  bool uniform, done, last_cta;

  // Balanced mode: the CTA's position range and first sequence, found once per CTA at
  // kernel start (balanced_range) and read from shared memory by every role.
  __device__ void init(const DecodeParams& p, int c, const SharedState* sh) {
    cta = c;
    done = false;
    if (p.num_splits >= 1) {
      uniform = true;
      ns = p.num_splits;
      b = c / ns;
      split = c % ns;
      return;
    }
    uniform = false;
    int Ge = balanced_ctas(sh->seg_total, p.num_ctas);
    if (c >= Ge) { done = true; return; }
    lo = sh->seg_lo;
    hi = sh->seg_hi;
    last_cta = (c == Ge - 1);
    b = sh->seg_b0;
  }

  __device__ bool next(const DecodeParams& p, Seg& s) {
    if (done) return false;
    if (uniform) {
      int r0;
      long long L;
      int rows = 1;
      if constexpr (PG) {
        // b is a query row.  Several query tokens per sequence (qo_indptr): row b is token
        // t of the q_len tokens of sequence sb and sees the first L - q_len + 1 + t tokens.
        int sb = b;
        if (p.qo_indptr != nullptr) {   // largest sb with qo_indptr[sb] <= b
          int lo = 0, hi = p.num_seqs - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.qo_indptr[mid] <= b) lo = mid; else hi = mid - 1;
          }
          sb = lo;
        }
        r0 = p.kv_indptr[sb];           // the sequence's first entry in the page list
        L = static_cast<long long>(p.kv_indptr[sb + 1]) - r0;
        L = L > 0 ? (L - 1) * p.page_size + p.last_page_len[sb] : 0;
        if (p.qo_indptr != nullptr) {
          const int qn = p.qo_indptr[sb + 1] - p.qo_indptr[sb];
          int t0 = b - p.qo_indptr[sb], last = t0;
          if (p.pair_rows) {
            // Fused instances: the CTAs of an even-numbered token t0 decode tokens t0 and
            // t0 + 1 together (their segment is the visible range of the later one); those
            // of an odd-numbered token have no work.
            if (t0 & 1) { done = true; return false; }
            if (t0 + 1 < qn) last = t0 + 1;
            rows = last - t0 + 1;
          }
          L -= qn - 1 - last;
          if (L < 0) L = 0;
        }
      } else {
        r0 = p.kv_indptr[b];
        L = static_cast<long long>(p.kv_indptr[b + 1]) - r0;
      }
      long long per = (L + ns - 1) / ns;
      long long chunk = ((per + kBN - 1) / kBN) * kBN;
      long long a = split * chunk, e = a + chunk;
      if (a > L) a = L;
      if (e > L) e = L;
      s.rows = rows; s.b = b; s.row0 = r0; s.n_lo = (int)a; s.n_hi = (int)e; s.n_total = (int)L;
      s.slot = b * ns + split; s.direct = (ns == 1);
      done = true;
      return true;
    }
    // Non-empty sequences: the part inside [lo, hi).  An empty sequence at token position x
    // belongs to the CTA with lo <= x < hi (the last CTA also owns x == total); it is
    // returned as an empty direct segment so that its output row gets written as zeros.
    while (b < p.batch) {
      // [r0, r1): the sequence's positions (paged: its tokens in the page space; the rest
      // of its last page belongs to no sequence).  row0: its first cache row (paged: its
      // first page-list entry).
      using Pos = typename std::conditional<PG, long long, int>::type;
      Pos r0 = p.kv_indptr[b], r1 = p.kv_indptr[b + 1];
      const int row0 = static_cast<int>(r0);
      if constexpr (PG) {
        r1 = r1 > r0 ? r0 * p.page_size + (r1 - r0 - 1) * p.page_size + p.last_page_len[b] : r0 * p.page_size;
        r0 *= p.page_size;
      }
      if (r0 > hi || (r0 == hi && !last_cta)) break;
      int bb = b++;
      if (r1 > r0) {
        long long a = lo > r0 ? lo : r0, e = hi < r1 ? hi : r1;
        if (e > a) {
          s.rows = 1; s.b = bb; s.row0 = row0; s.n_lo = (int)(a - r0); s.n_hi = (int)(e - r0); s.n_total = (int)(r1 - r0);
          s.slot = bb + cta; s.direct = (a == r0 && e == r1);
          return true;
        }
      } else if (r0 >= lo && (r0 < hi || last_cta)) {
        s.rows = 1; s.b = bb; s.row0 = row0; s.n_lo = 0; s.n_hi = 0; s.n_total = 0; s.slot = bb + cta; s.direct = true;
        return true;
      }
    }
    done = true;
    return false;
  }
};

// The 128-row TMA window of tile t of a segment.  The window never extends past the
// segment's last row (it is shifted back instead; rows before 0 are zero-filled by TMA),
// so the kernel reads no row outside [0, kv_indptr[batch]).
struct Window {
  int y0;     // first cached row of the window (may be negative; paged: unused)
  int shift;  // window row of the tile's first token
  int cnt;    // valid tokens in the tile
};
// Contiguous cache: the window ends at the segment's last row (rows before cached row 0 are
// the TMA's zero fill).  Paged cache: tiles start on page boundaries (the segment starts on
// one, a tile is 128 tokens and the page size divides 128), window row i is token start + i
// of the sequence, and the rows come from the pages (paged_entry); shift is 0.
// Page-list entry holding window row i of tile t (the sequence's last page again for rows
// past its end, which are masked).
// (Page arithmetic by shifts: page_size is a power of two, page_shift its log2.)
template <bool PG>
__device__ __forceinline__ int paged_entry(const DecodeParams& p, const Seg& s, int t, int i) {
  const int np = (s.n_total + p.page_size - 1) >> p.page_shift;
  return p.page_indices[s.row0 + min((s.n_lo + t * kBN + i) >> p.page_shift, np - 1)];
}
template <int KV, bool PG>
__device__ __forceinline__ Window tile_window(const DecodeParams& p, const Seg& s, int t) {
  Window w;
  if constexpr (PG) {
    const int start = s.n_lo + t * kBN;
    w.y0 = 0;
    w.shift = 0;
    w.cnt = min(kBN, s.n_hi - start);
  } else {
    int row_start = s.row0 + s.n_lo + t * kBN;
    int row_hi = s.row0 + s.n_hi;
    int y0 = min(row_start, row_hi - kBN);
    w.y0 = y0;
    w.shift = row_start - y0;
    w.cnt = min(kBN, row_hi - row_start);
  }
  return w;
}

__device__ __forceinline__ float bf16_bits_to_f(uint32_t b) { return __uint_as_float(b << 16); }

// 2^n exactly, for -149 <= n <= 127, from the exponent bits (subnormal below 2^-126).
__device__ __forceinline__ float pow2i(int n) {
  return n >= -126 ? __uint_as_float(static_cast<uint32_t>(n + 127) << 23) : __uint_as_float(1u << (n + 149));
}

__device__ __forceinline__ uint16_t f_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 unpack_e4m3x2(uint32_t v) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xFFFFu), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __half22float2(h);
}

// One arrival per warp on an mbarrier whose count is in warps: the lanes' earlier shared
// memory writes (and their proxy / tcgen05 fences) are ordered before lane 0's arrive by
// the warp barrier.  Called by all 32 lanes.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// ---------------------------------------------------------------- q staging
// bf16: Q[16 x 576] -> 9 K-major SW128 chunks [16 QL rows x 128 B]; query token j (staged by
// threads 128 j .. 128 j + 127) fills rows 16 j .. 16 j + 15 of every chunk (zeros when the
// token does not exist: `rows` query rows are staged).
template <int QL>
__device__ void stage_q_bf16(const DecodeParams& p, int b, int rows, uint8_t* qs, int ts) {
  const int tok = ts >> 7, t = ts & 127;
  const uint4* src = reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(b + tok) * kHeads * kDim);
  for (int i = t; i < kHeads * 72; i += 128) {
    int h = i / 72, pc = i % 72;
    int c = pc >> 3, j = pc & 7;
    const int r = 16 * tok + h;
    uint4 v = tok < rows ? __ldg(src + h * 72 + pc) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(qs + c * 2048 * QL + r * 128 + ((j ^ (r & 7)) << 4)) = v;
  }
}

// fp8 path: per head h, q*2^a_h = hi + lo/16 with hi, lo e4m3 (exact for every bf16 q whose
// scaled magnitude is >= 2^-6; a_h puts the head's max near 2^8).  For query token j (staged
// by threads 128 j .. 128 j + 127), rows 32 j + 0..15 of each [32 QL x 128 B] chunk hold hi
// and rows 32 j + 16..31 hold lo; qscale[16 j + h] = 2^-a_h.  A token that does not exist
// (j >= rows) is staged as zeros.
template <int QL>
__device__ void stage_q_fp8(const DecodeParams& p, int b, int rows, uint8_t* qs, float* qscale, int ts) {
  const int tok = ts >> 7;
  const int h = (ts & 127) >> 3, t8 = ts & 7;
  const uint4* src =
      reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b + tok) * kHeads + h) * kDim + 72 * t8);
  uint4 v[9];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    v[i] = tok < rows ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f(w[k] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f(w[k] >> 16)));
    }
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  int e = 0;
  frexpf(amax, &e);
  const int a = amax > 0.f ? min(max(8 - e, -126), 126) : 0;
  const float sc = pow2i(a);
  if (t8 == 0) qscale[16 * tok + h] = pow2i(-a);
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
      float y0 = bf16_bits_to_f(w[k] & 0xFFFFu) * sc, y1 = bf16_bits_to_f(w[k] >> 16) * sc;
      float y2 = bf16_bits_to_f(w[k + 1] & 0xFFFFu) * sc, y3 = bf16_bits_to_f(w[k + 1] >> 16) * sc;
      uint32_t h01 = pack_e4m3x2(y0, y1), h23 = pack_e4m3x2(y2, y3);
      float2 d01 = unpack_e4m3x2(h01), d23 = unpack_e4m3x2(h23);
      uint32_t l01 = pack_e4m3x2((y0 - d01.x) * 16.f, (y1 - d01.y) * 16.f);
      uint32_t l23 = pack_e4m3x2((y2 - d23.x) * 16.f, (y3 - d23.y) * 16.f);
      hi[k >> 1] = h01 | (h23 << 16);
      lo[k >> 1] = l01 | (l23 << 16);
    }
    const int f0 = 72 * t8 + 8 * i;
    const int c = f0 >> 7, jb = f0 & 127, piece = jb >> 4, half = (jb >> 3) & 1;
    const int rh = 32 * tok + h, rl = rh + 16;
    if (c < 4) {   // value dims: [32 QL rows x 128 B] SW128 chunks
      const int off = ((piece ^ (h & 7)) << 4) + half * 8;
      *reinterpret_cast<uint2*>(qs + c * 4096 * QL + rh * 128 + off) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(qs + c * 4096 * QL + rl * 128 + off) = make_uint2(lo[0], lo[1]);
    } else {       // rope dims: [32 QL rows x 64 B] SW64
      *reinterpret_cast<uint2*>(qs + 4 * 4096 * QL + rh * 64 + ((piece ^ ((rh >> 1) & 3)) << 4) + half * 8) =
          make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(qs + 4 * 4096 * QL + rl * 64 + ((piece ^ ((rl >> 1) & 3)) << 4) + half * 8) =
          make_uint2(lo[0], lo[1]);
    }
  }
}

// ---------------------------------------------------------------- producer (1 thread)
// MXFP4: each tile is fetched as five column slabs of the packed rows (2D TMA, 64-byte
// boxes, 64-byte swizzle): bytes [64c, 64c + 64) of the window's 128 rows for the value
// chunks c = 0..3 and bytes [256, 288) for the rope chunk (the box's columns past 288 are
// zero-filled).  The dequantisation frees each slab as soon as it has read it.
// Paged producers run on the whole warp: lane k < 128/P owns page k of the tile (one TMA
// box of P rows, at window row k P).  Its physical first row, loaded once per tile:
template <bool PG>
__device__ __forceinline__ int lane_page_row(const DecodeParams& p, const Seg& s, int t, int lane) {
  const int nb = kBN >> p.page_shift;
  const int np = (s.n_total + p.page_size - 1) >> p.page_shift;
  const int pg = min(((s.n_lo + t * kBN) >> p.page_shift) + min(lane, nb - 1), np - 1);
  return p.page_indices[s.row0 + pg] << p.page_shift;
}
// Issues the boxes of one slot: the whole 128-row window (contiguous, one lane) or one box
// per page (paged, lane k: box k lands k * bytes * P / 128 bytes into the slot, a multiple
// of the swizzle atom for P >= 8).
template <bool PG>
__device__ __forceinline__ void load_window(const DecodeParams& p, const CUtensorMap* map, uint32_t dst, int x,
                                            uint32_t bytes, int y0, int lane, int lane_row, uint32_t fb) {
  if constexpr (PG) {
    static_assert(kBN == 128, "bytes * P / 128 below assumes 128-row tiles");
    if (lane < (kBN >> p.page_shift)) tma_load_2d(dst + ((lane * bytes) >> (7 - p.page_shift)), map, x, lane_row, fb);
  } else {
    tma_load_2d(dst, map, x, y0, fb);
  }
}
// Sets the slot's expected bytes: one lane (contiguous) or lane 0 of the paged warp, before
// any lane issues a box.
template <bool PG>
__device__ __forceinline__ void expect_slot(uint32_t fb, uint32_t bytes, int lane) {
  if constexpr (PG) {
    if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
    __syncwarp();
  } else {
    mbar_arrive_expect_tx(fb, bytes);
  }
}
// The warp-wide (paged) producer agrees on every wait's outcome.
template <bool PG>
__device__ __forceinline__ bool producer_wait(uint32_t bar, uint32_t parity, volatile int* abortf, int* status,
                                              uint64_t limit) {
  const bool ok = wait_bar(bar, parity, abortf, status, limit);
  if constexpr (PG) return __all_sync(0xffffffffu, ok);
  return ok;
}

template <bool PG>
__device__ void run_producer_mx(const DecodeParams& p, SharedState* sh, uint8_t* slabs, int lane) {
  volatile int* abortf = &sh->abort;
  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t idx = 0, slot = 0, phase = 0;
  bool ok = true;
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    const int ntiles = (n + kBN - 1) / kBN;
    for (int t = 0; t < ntiles && ok; ++t) {
      const Window w = tile_window<2, PG>(p, s, t);
      int lrow = 0;
      if constexpr (PG) lrow = lane_page_row<PG>(p, s, t, lane);
      for (int i = 0; i < 5; ++i) {
        const int c = mx_chunk(i);
        if (!producer_wait<PG>(smem_u32(&sh->slab_empty[slot]), phase ^ 1, abortf, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh->slab_full[slot]);
        expect_slot<PG>(fb, kSlabBytes, lane);
        load_window<PG>(p, &p.tmap, smem_u32(slabs + slot * kSlabBytes), 64 * c, kSlabBytes, w.y0, lane, lrow, fb);
        ++idx;
        if (++slot == kSlabs) { slot = 0; phase ^= 1; }
      }
    }
  }
  if (!ok) {  // drain copies already issued so that none lands after the CTA exits
    const uint32_t first = idx > (uint32_t)kSlabs ? idx - kSlabs : 0u;
    for (uint32_t j = first; j < idx; ++j)
      wait_bar(smem_u32(&sh->slab_full[j % kSlabs]), (j / kSlabs) & 1, abortf, p.status, kDrainLimitNs, false);
  }
}

template <int KV, bool PG, int QL>
__device__ void run_producer(const DecodeParams& p, SharedState* sh, uint8_t* ring, uint8_t* rope, int lane) {
  using C = Cfg<KV>;
  constexpr int kRing = Geo<KV, QL>::kRing;
  volatile int* abortf = &sh->abort;
  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t idx = 0, slot = 0, phase = 0, ridx = 0;
  bool ok = true;
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    const int ntiles = (n + kBN - 1) / kBN;
    for (int t = 0; t < ntiles && ok; ++t) {
      const Window w = tile_window<KV, PG>(p, s, t);
      int lrow = 0;
      if constexpr (PG) lrow = lane_page_row<PG>(p, s, t, lane);
      for (int c = 0; c < C::kRingPT; ++c) {
        if (!producer_wait<PG>(smem_u32(&sh->empty[slot]), phase ^ 1, abortf, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(ring + slot * C::kSlotBytes);
        const uint32_t fb = smem_u32(&sh->full[slot]);
        auto box = [&](uint32_t d, int x, uint32_t bytes) { load_window<PG>(p, &p.tmap, d, x, bytes, w.y0, lane, lrow, fb); };
        if constexpr (KV == 0) {
          if (c < 4) {
            expect_slot<PG>(fb, 32768, lane);
            box(dst, 128 * c, 16384);
            box(dst + 16384, 128 * c + 64, 16384);
          } else {
            expect_slot<PG>(fb, 16384, lane);
            box(dst, 512, 16384);
          }
        } else {
          expect_slot<PG>(fb, 16384, lane);
          box(dst, 128 * c, 16384);
        }
        ++idx;
        if (++slot == kRing) { slot = 0; phase ^= 1; }
      }
      if constexpr (C::kRopeSlots > 0) {   // fp8: the rope chunk (64 B of each row) into its own slots
        if (!ok) break;
        const uint32_t rs = ridx % C::kRopeSlots;
        if (!producer_wait<PG>(smem_u32(&sh->rope_empty[rs]), ((ridx / C::kRopeSlots) & 1) ^ 1, abortf, p.status,
                               p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh->rope_full[rs]);
        expect_slot<PG>(fb, kRopeBytes, lane);
        load_window<PG>(p, &p.tmap_rope, smem_u32(rope + rs * kRopeBytes), kDimV, kRopeBytes, w.y0, lane, lrow, fb);
        ++ridx;
      }
    }
  }
  if (!ok) {  // drain copies already issued so that none lands after the CTA exits
    const uint32_t first = idx > (uint32_t)kRing ? idx - kRing : 0u;
    for (uint32_t j = first; j < idx; ++j)
      wait_bar(smem_u32(&sh->full[j % kRing]), (j / kRing) & 1, abortf, p.status, kDrainLimitNs, false);
    if constexpr (C::kRopeSlots > 0) {
      const uint32_t rfirst = ridx > (uint32_t)C::kRopeSlots ? ridx - C::kRopeSlots : 0u;
      for (uint32_t j = rfirst; j < ridx; ++j)
        wait_bar(smem_u32(&sh->rope_full[j % C::kRopeSlots]), (j / C::kRopeSlots) & 1, abortf, p.status,
                 kDrainLimitNs, false);
    }
  }
}

// ---------------------------------------------------------------- producer for pages of 1-4 rows (1 warp)
// A tiled TMA box of fewer than 8 rows would not fill whole 8-row swizzle atoms, so bf16 and
// fp8 pages of 1, 2 or 4 rows are fetched with four-row gathers (tile::gather4) from maps
// whose box is one row high: lane k gathers window rows 4k..4k+3 (their cache rows through
// the page list) to rows 4k..4k+3 of the slot, where the copy engine swizzles each row by its
// own shared address, as a 128-row box would be laid out.  Lane 0 sets the slot's expected
// bytes first; the slot completes on bytes, like the tiled loads.  (MXFP4 slabs: cp.async,
// below.)
// MXFP4 slabs are 64 bytes wide, and a gather of four such rows moves too little per copy
// engine operation: their pages of 1-4 rows are copied with 16-byte cp.async straight into
// the slab's SW64 layout instead (piece j of window row r at r * 64 + ((j ^ (r / 2) mod 4)
// << 4)), every lane arriving on the slab's full barrier when its own copies have landed.
// Bytes [byte0, byte0 + W) of each of the tile's 128 window rows, whose cache rows are in
// `rows`; lane = (row, piece) so that each warp-wide copy reads whole 32-byte sectors.
template <int W, int PITCH>
__device__ __forceinline__ void sp_copy(const uint8_t* kv, int row_bytes, const int* rows, uint32_t dst, int byte0,
                                        int lane) {
  constexpr int kPieces = W / 16;
  constexpr int kRowsPer = 32 / kPieces;
  const int piece = lane % kPieces;
#pragma unroll 4
  for (int r = lane / kPieces; r < kBN; r += kRowsPer) {
    const uint8_t* src = kv + static_cast<size_t>(rows[r]) * row_bytes + byte0 + piece * 16;
    const int sw = PITCH == 128 ? (r & 7) : ((r >> 1) & 3);
    cp_async_16(dst + r * PITCH + ((piece ^ sw) << 4), src);
  }
}

template <int KV, int QL>
__device__ void run_producer_sp(const DecodeParams& p, SharedState* sh, uint8_t* ring, uint8_t* rope, uint8_t* slabs,
                                int lane) {
  using C = Cfg<KV>;
  volatile int* abortf = &sh->abort;
  SegIter<true> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t idx = 0, slot = 0, phase = 0, ridx = 0;
  constexpr int kSlots = KV == 2 ? kSlabs : Geo<KV, QL>::kRing;
  bool ok = true;
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    const int ntiles = (n + kBN - 1) / kBN;
    const int np = (s.n_total + p.page_size - 1) >> p.page_shift;
    for (int t = 0; t < ntiles && ok; ++t) {
      // Cache rows of this lane's four window rows (rows past the sequence reuse its last
      // page; they are masked).  MXFP4: every window row's, in shared memory for sp_copy.
      int y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = s.n_lo + t * kBN + 4 * lane + i;
        y[i] = (p.page_indices[s.row0 + min(tok >> p.page_shift, np - 1)] << p.page_shift) + (tok & (p.page_size - 1));
      }
      if constexpr (KV == 2) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) sh->sp_rows[4 * lane + i] = y[i];
        __syncwarp();
      }
      // Four rows of `pitch` bytes per lane at column x of `map`, into the slot image at dst.
      auto gather = [&](uint32_t dst, const CUtensorMap* map, int x, int pitch, uint32_t fb) {
        tma_gather4(dst + 4 * lane * pitch, map, x, y[0], y[1], y[2], y[3], fb);
      };
      for (int c0 = 0; c0 < (KV == 2 ? 5 : C::kRingPT); ++c0) {
        const uint32_t eb = KV == 2 ? smem_u32(&sh->slab_empty[slot]) : smem_u32(&sh->empty[slot]);
        if (!producer_wait<true>(eb, phase ^ 1, abortf, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        if constexpr (KV == 2) {
          const int c = mx_chunk(c0);
          const uint32_t dst = smem_u32(slabs + slot * kSlabBytes);
          if (c < 4) sp_copy<64, 64>(p.kv, kMxPacked, sh->sp_rows, dst, 64 * c, lane);
          else sp_copy<32, 64>(p.kv, kMxPacked, sh->sp_rows, dst, 4 * 64, lane);   // the rope's 32 bytes (the rest unused)
          cp_async_mbar_arrive(smem_u32(&sh->slab_full[slot]));
        } else {
          const uint32_t dst = smem_u32(ring + slot * C::kSlotBytes);
          const uint32_t fb = smem_u32(&sh->full[slot]);
          if constexpr (KV == 0) {   // x in bf16 elements; value slots hold two 64-column boxes
            if (c0 < 4) {
              expect_slot<true>(fb, 32768, lane);
              gather(dst, &p.tmap, 128 * c0, 128, fb);
              gather(dst + 16384, &p.tmap, 128 * c0 + 64, 128, fb);
            } else {
              expect_slot<true>(fb, 16384, lane);
              gather(dst, &p.tmap, kDimV, 128, fb);
            }
          } else {
            expect_slot<true>(fb, 16384, lane);
            gather(dst, &p.tmap, 128 * c0, 128, fb);
          }
        }
        ++idx;
        if (++slot == static_cast<uint32_t>(kSlots)) { slot = 0; phase ^= 1; }
      }
      if constexpr (KV == 1) {   // the rope chunk (64 B of each row) into its own slots
        if (!ok) break;
        const uint32_t rs = ridx % C::kRopeSlots;
        if (!producer_wait<true>(smem_u32(&sh->rope_empty[rs]), ((ridx / C::kRopeSlots) & 1) ^ 1, abortf, p.status,
                                 p.wait_limit_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh->rope_full[rs]);
        expect_slot<true>(fb, kRopeBytes, lane);
        gather(smem_u32(rope + rs * kRopeBytes), &p.tmap_rope, kDimV, 64, fb);
        ++ridx;
      }
    }
  }
  if (!ok) {  // drain copies already issued so that none lands after the CTA exits
    const uint32_t first = idx > static_cast<uint32_t>(kSlots) ? idx - kSlots : 0u;
    for (uint32_t j = first; j < idx; ++j) {
      const uint32_t fb = KV == 2 ? smem_u32(&sh->slab_full[j % kSlots]) : smem_u32(&sh->full[j % kSlots]);
      wait_bar(fb, (j / kSlots) & 1, abortf, p.status, kDrainLimitNs, false);
    }
    if constexpr (KV == 1) {
      const uint32_t rfirst = ridx > (uint32_t)C::kRopeSlots ? ridx - C::kRopeSlots : 0u;
      for (uint32_t j = rfirst; j < ridx; ++j)
        wait_bar(smem_u32(&sh->rope_full[j % C::kRopeSlots]), (j / C::kRopeSlots) & 1, abortf, p.status,
                 kDrainLimitNs, false);
    }
  }
}

// ---------------------------------------------------------------- MXFP4 dequantisation (128 threads)
// Row i of a tile (thread i) becomes 576 e4m3 carrier bytes: block j of 32 elements is
// e2m1 * 2^(E_j - e_i) with e_i = max_j E_j, looked up per nibble in an 8-entry table for
// the shift E_j - e_i (exact for shifts >= -8, e4m3-rounded below, zero below -12).
// The row factor 2^(e_i - 127) is applied by the softmax to the logits and to P.
// Layout: the same K-major SW128 chunks the TMA writes for fp8 caches (value chunks) and
// a [128 x 64 B] SW64 buffer for the rope chunk.

// Byte permute with sign replication (PTX prmt default mode: a selector nibble with its
// top bit set yields the selected byte's top bit copied into all eight bits).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// Eight e2m1 nibbles (one packed word, element k in bits 4k..4k+3) -> eight e4m3 bytes:
// magnitudes through the shift table (byte permute on the 3-bit codes); each element's
// sign bit (bit 3 of its nibble) is the top bit of a byte of w (odd elements) or of w << 4
// (even elements), so one sign-replicating permute per four elements yields its sign mask.
__device__ __forceinline__ void e2m1x8_to_e4m3x8(uint32_t w, uint2 lut, uint32_t& lo, uint32_t& hi) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t w4 = w << 4;
  lo = prmt(lut.x, lut.y, m) | (prmt(w4, w, 0xD9C8u) & 0x80808080u);
  hi = prmt(lut.x, lut.y, m >> 16) | (prmt(w4, w, 0xFBEAu) & 0x80808080u);
}
// One 32-element block (16 packed bytes) -> 32 carrier bytes (two 16-byte pieces).
__device__ __forceinline__ void deq_block(const uint4 v, const uint2 lut, uint4& lo, uint4& hi) {
  e2m1x8_to_e4m3x8(v.x, lut, lo.x, lo.y);
  e2m1x8_to_e4m3x8(v.y, lut, lo.z, lo.w);
  e2m1x8_to_e4m3x8(v.z, lut, hi.x, hi.y);
  e2m1x8_to_e4m3x8(v.w, lut, hi.z, hi.w);
}

// Tile g, chunk c: the packed bytes come from slab 5g + c of the slab ring; value chunk c
// (128 dims) goes to ring slot 4 * (g & 1) + c (the ring holds the value chunks of exactly
// two tiles, so dequantising tile g + 2 only waits for the PV MMAs of tile g); the rope
// chunk goes to its own SW64 buffer and is published (and its slab freed) as soon as it is
// done; the four value chunks are published (on the last one's barrier, the one the QK
// issuer waits for), and their slabs freed, together.  Window rows
// before cached row 0 hold zeros (TMA fill) and get no scale: they decode to zeros.
template <bool PG>
__device__ void run_dequant(const DecodeParams& p, SharedState* sh, uint8_t* ring, uint8_t* rope, uint8_t* slabs) {
  using C = Cfg<2>;
  volatile int* abortf = &sh->abort;
  const int dt = threadIdx.x - 32 * (4 + C::kSoftWarps);   // dequant thread
  const int di = dt % kBN;                                 // carrier row of the tile
  // With kRowThreads = 2, thread half hh converts blocks {2 hh, 2 hh + 1} of each 4-block
  // value chunk and block hh of the rope chunk.
  constexpr int kRT = C::kRowThreads;
  const int hh = dt / kBN;
  const uint8_t* scales = static_cast<const uint8_t*>(p.kv_scale);
  if (dt < kLutCount * 8) {
    const int k = dt >> 3, c = dt & 7;
    const float mag = (c < 2) ? 0.5f * c : ldexpf(1.0f + 0.5f * (c & 1), (c >> 1) - 1);
    const uint32_t code = (k >= 13) ? 0u
        : static_cast<uint32_t>(__nv_cvt_float_to_fp8(ldexpf(mag, -k), __NV_SATFINITE, __NV_E4M3));
    reinterpret_cast<uint8_t*>(&sh->lut[0])[k * 8 + c] = static_cast<uint8_t>(code);
  }
  bar_sync(2, C::kDeqWarps * 32);
  const int ssw = (di >> 1) & 3;           // SW64 piece swizzle of this row in a slab
  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t g = 0, slab_i = 0, slab_ph = 0;
  bool ok = true;
  // Barrier tests issued ahead of the work they gate (their shared-memory round trips overlap
  // the conversion; a test that finds the phase incomplete falls back to the bounded wait).
  bool pre_slab = false;   // the next slab to read has landed
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    const int ntiles = (n + kBN - 1) / kBN;
    uint32_t scn[9];   // block scales of the segment's next tile, loaded one tile ahead
    for (int t = 0; t < ntiles; ++t) {
      // Rope carrier slot g mod 2 was last read by the QK MMAs of tile g - 2; the value slots
      // by the PV MMAs of tile g - 2.
      const bool pre_rope = mbar_test_wait(smem_u32(&sh->rope_empty[g & 1]), ((g >> 1) & 1) ^ 1);
      const bool pre_pv = g < 2 || mbar_test_wait(smem_u32(&sh->pv_done[g & 1]), ((g >> 1) & 1) ^ 1);
      const Window w = tile_window<2, PG>(p, s, t);
      // e_i = max_j E_j and the shift-table index min(e_i - E_j, 13) of each block, packed
      // as 4-bit fields (block j in bits 4 (j % 8) of kpk[j / 8]).
      int emax = 127;
      uint32_t kpk[3] = {0u, 0u, 0u};
      // Cached row of this thread's window row (paged: its page's physical row).
      const int yr = PG ? (paged_entry<PG>(p, s, t, di) << p.page_shift) + (di & (p.page_size - 1)) : w.y0 + di;
      if (yr >= 0) {
        uint32_t sc[9];
        if (t > 0) {
#pragma unroll
          for (int j = 0; j < 9; ++j) sc[j] = scn[j];
        } else {
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(scales + static_cast<size_t>(yr) * kMxScales);
#pragma unroll
          for (int j = 0; j < 9; ++j) sc[j] = __ldg(sp + j);
        }
        // The row exponent never goes below kRowExpFloor: a row whose blocks all sit below
        // 2^(kRowExpFloor - 127) (an all-zero row with e8m0 code 0, for instance) keeps a
        // PV weight 2^(logit + e_i - 127) inside fp32's normal range.
        emax = kRowExpFloor;
#pragma unroll
        for (int j = 0; j < 9; ++j) emax = max(emax, max(static_cast<int>(sc[j] & 0xFF), static_cast<int>(sc[j] >> 8)));
#pragma unroll
        for (int j = 0; j < 18; ++j) {
          const int e = static_cast<int>((sc[j >> 1] >> (8 * (j & 1))) & 0xFF);
          kpk[j >> 3] |= static_cast<uint32_t>(min(emax - e, kLutCount - 1)) << (4 * (j & 7));
        }
      }
      if (t + 1 < ntiles) {
        const Window wn = tile_window<2, PG>(p, s, t + 1);
        const int yn = PG ? (paged_entry<PG>(p, s, t + 1, di) << p.page_shift) + (di & (p.page_size - 1)) : wn.y0 + di;
        if (yn >= 0) {
          const uint16_t* sp = reinterpret_cast<const uint16_t*>(scales + static_cast<size_t>(yn) * kMxScales);
#pragma unroll
          for (int j = 0; j < 9; ++j) scn[j] = __ldg(sp + j);
        }
      }
      // Fully unrolled over the 18 blocks so that the block indices are constants.
      // Rolled over the five chunks (the loop body holds one value chunk and the rope chunk),
      // so that the dequantisation code stays small next to the softmax and issue loops
      // sharing the SM's instruction cache.  Shift-table indices of blocks 0-15 come from
      // one 64-bit register by a run-time shift.
      const uint64_t kv64 = static_cast<uint64_t>(kpk[0]) | (static_cast<uint64_t>(kpk[1]) << 32);
      // The rope chunk comes first (the producer fetches it first and the QK MMAs take it
      // first): its carrier slot (one of two) was last read by the QK MMAs of tile g - 2, so
      // it does not wait for the PV MMAs of tile g - 2, which the value chunks below do.
      {
        const uint32_t si = slab_i, sph = slab_ph;
        if (++slab_i == kSlabs) { slab_i = 0; slab_ph ^= 1u; }
        if (!__all_sync(0xffffffffu, pre_slab)) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&sh->slab_full[si]), sph, abortf, p.status, p.wait_limit_ns));
          if (!ok) break;
        }
        const uint32_t srow = smem_u32(slabs + si * kSlabBytes + di * 64);
        uint4 v0, v1;
        if constexpr (kRT == 1) {
          v0 = ld_shared_v4_volatile(srow + ((0 ^ ssw) << 4));
          v1 = ld_shared_v4_volatile(srow + ((1 ^ ssw) << 4));
        } else {
          v0 = ld_shared_v4_volatile(srow + ((hh ^ ssw) << 4));
        }
        // The slab goes back to the producer as soon as it has been read.  Its next fill is
        // an async-proxy (TMA) write to the bytes these generic-proxy loads just read, and
        // the mbarrier hand-off alone does not order the two proxies: the proxy fence comes
        // first.  (Without it, about one balanced-mode call in twenty with one- or two-tile
        // segments read a few MX blocks of a value chunk from the slab's next fill.)
        fence_proxy_async_smem();
        warp_arrive(smem_u32(&sh->slab_empty[si]));
        pre_slab = mbar_test_wait(smem_u32(&sh->slab_full[slab_i]), slab_ph);   // value chunk 0's slab
        if (!__all_sync(0xffffffffu, pre_rope)) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&sh->rope_empty[g & 1]), ((g >> 1) & 1) ^ 1, abortf,
                                                p.status, p.wait_limit_ns));
          if (!ok) break;
        }
        uint8_t* dst = rope + (g & 1) * kRopeBytes + di * 64;                 // [128 x 64 B] SW64
        uint4 lo, hi;
        if constexpr (kRT == 1) {
          deq_block(v0, sh->lut[kpk[2] & 15u], lo, hi);
          *reinterpret_cast<uint4*>(dst + ((0 ^ ssw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + ((1 ^ ssw) << 4)) = hi;
          deq_block(v1, sh->lut[(kpk[2] >> 4) & 15u], lo, hi);
          *reinterpret_cast<uint4*>(dst + ((2 ^ ssw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + ((3 ^ ssw) << 4)) = hi;
        } else {
          deq_block(v0, sh->lut[(kpk[2] >> (4 * hh)) & 15u], lo, hi);
          *reinterpret_cast<uint4*>(dst + (((2 * hh) ^ ssw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * hh + 1) ^ ssw) << 4)) = hi;
        }
        if (hh == 0) sh->etok[g & 3][di] = emax;
        fence_proxy_async_smem();
        warp_arrive(smem_u32(&sh->rope_full[g & 1]));
      }
      // The value slots of tile g were last read by tile g - 2: one wait on its PV completion
      // covers all four (QK of g - 2 completed before its softmax, hence before its PV).
      static_assert(C::kRing == 2 * C::kRingPT, "the MXFP4 value ring holds exactly two tiles");
      if (!__all_sync(0xffffffffu, pre_pv)) {
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&sh->pv_done[g & 1]), ((g >> 1) & 1) ^ 1, abortf, p.status,
                                              p.wait_limit_ns));
        if (!ok) break;
      }
      const uint32_t vslot0 = (g & 1) * C::kRingPT;
      // The four value chunks are converted back to back and handed over together: one proxy
      // fence orders this thread's generic reads of the four slabs (before their next
      // async-proxy fills) and its carrier stores (before the MMAs read them), then the four
      // slabs go back to the producer and the four chunks are published.  The QK MMAs of a
      // tile wait for its last chunk in any case.
      const uint32_t si0 = slab_i;
#pragma unroll 1
      for (int c = 0; c < C::kRingPT; ++c) {
        const uint32_t si = slab_i, sph = slab_ph;
        if (++slab_i == kSlabs) { slab_i = 0; slab_ph ^= 1u; }
        if (!__all_sync(0xffffffffu, pre_slab)) {
          ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&sh->slab_full[si]), sph, abortf, p.status, p.wait_limit_ns));
          if (!ok) break;
        }
        // The packed words are read with volatile loads, which ptxas schedules better here
        // (256 x 8192: 376 -> 345 us).
        const uint32_t srow = smem_u32(slabs + si * kSlabBytes + di * 64);
        constexpr int kB = 4 / kRT;                                           // blocks per thread
        const int b0 = kRT == 1 ? 0 : kB * hh;
        uint4 v[kB];
#pragma unroll
        for (int q = 0; q < kB; ++q) v[q] = ld_shared_v4_volatile(srow + (((b0 + q) ^ ssw) << 4));
        // The next slab: value chunk c + 1, or the next tile's rope chunk.
        pre_slab = mbar_test_wait(smem_u32(&sh->slab_full[slab_i]), slab_ph);
        uint8_t* dst = ring + (vslot0 + c) * C::kSlotBytes + di * 128;       // [128 x 128 B] SW128
        const uint32_t kc = static_cast<uint32_t>(kv64 >> (16 * c + 4 * b0)); // blocks 4c + b0 ..
#pragma unroll
        for (int q = 0; q < kB; ++q) {
          const int bk = b0 + q;
          uint4 lo, hi;
          deq_block(v[q], sh->lut[(kc >> (4 * q)) & 15u], lo, hi);
          *reinterpret_cast<uint4*>(dst + (((2 * bk) ^ (di & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * bk + 1) ^ (di & 7)) << 4)) = hi;
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
#pragma unroll
      for (int c = 0; c < C::kRingPT; ++c) warp_arrive(smem_u32(&sh->slab_empty[(si0 + c) % kSlabs]));
      // The QK MMAs take the four value chunks together, on the last chunk's barrier.
      warp_arrive(smem_u32(&sh->full[vslot0 + C::kRingPT - 1]));
      warp_arrive(smem_u32(&sh->etok_full[g & 3]));
      ++g;
    }
  }
}

// ---------------------------------------------------------------- MMA issuer (1 thread)
// MMA issue.  Single-thread issuers on separate warps keep the tensor core fed: one issues
// every QK^T group, two share the PV groups (two 128-dim blocks of O each; independent
// accumulators), each blocking only on its own barriers.  Shared-memory descriptors are built once; per MMA
// only the 14-bit start-address field advances (one 64-bit add), so an MMA costs a few
// instructions of issue.
struct Descs {
  uint64_t ring_k;   // K-major SW128 descriptor of ring slot 0 (sbo = 1024)
  uint64_t ring_mn;  // MN-major SW128 descriptor of ring slot 0 (lbo = 16 KB, sbo = 1024)
  uint64_t rope;     // K-major SW64 descriptor of the MXFP4 rope carrier (sbo = 512)
  uint64_t q;        // K-major SW128 descriptor of the q chunks
  uint64_t q_rope;   // K-major SW64 descriptor of the q rope chunk (fp8 / MXFP4)
  uint64_t p;        // MN-major SW32 descriptor of P buffer 0 (sbo = 256)
};
template <int QL>
__device__ __forceinline__ Descs make_descs(uint8_t* ring, uint8_t* rope, uint8_t* qs, uint8_t* ps) {
  Descs d;
  d.ring_k = smem_desc(smem_u32(ring), 16, 1024, kSwizzle128B);
  d.ring_mn = smem_desc(smem_u32(ring), 16384, 1024, kSwizzle128B);
  d.rope = smem_desc(smem_u32(rope), 16, 512, kSwizzle64B);
  d.q = smem_desc(smem_u32(qs), 16, 1024, kSwizzle128B);
  d.q_rope = smem_desc(smem_u32(qs + 4 * 4096 * QL), 16, 512, kSwizzle64B);
  // P^T rows are 32 QL bytes: one SW32 atom (QL = 1) or one SW64 atom (QL = 2) along N.
  d.p = QL == 1 ? smem_desc(smem_u32(ps), 0, 256, kSwizzle32B) : smem_desc(smem_u32(ps), 0, 512, kSwizzle64B);
  return d;
}
// Byte offset -> descriptor start-address increment.
__device__ __forceinline__ uint64_t dofs(uint32_t bytes) { return static_cast<uint64_t>(bytes >> 4); }

template <int KV, bool PG, bool SP, int QL>
__device__ void run_mma_qk(const DecodeParams& p, SharedState* sh, const Descs& ds, uint32_t tmem) {
  using C = Cfg<KV>;
  using G = Geo<KV, QL>;
  constexpr uint32_t idq = instr_desc(KV == 0 ? 1u : 0u, 0, 0, 128, G::kN);  // bf16 | e4m3, K-major A and B
  volatile int* abortf = &sh->abort;
  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t g = 0, slot = 0, phase = 0;
  int kseg = 0;
  // Test hook: a wait that can only end by running past the limit (status word, abort).
  bool ok = !p.test_stall || wait_bar(smem_u32(&sh->never), 0, abortf, p.status, p.wait_limit_ns);
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    ok = wait_bar(smem_u32(&sh->q_ready), kseg & 1, abortf, p.status, p.wait_limit_ns);
    const int ntiles = (n + kBN - 1) / kBN;
    for (int t = 0; ok && t < ntiles; ++t, ++g) {
      if (g >= 2 && !(ok = wait_bar(smem_u32(&sh->s_free[g & 1]), ((g >> 1) & 1) ^ 1, abortf, p.status,
                                    p.wait_limit_ns)))
        break;
      const uint32_t d = tmem + (g & 1) * G::kSCols;
#pragma unroll
      for (int i = 0; i < C::kSPT; ++i) {
        const int c = KV == 2 ? mx_chunk(i) : i;                             // MXFP4: the dequantisation order
        const bool rope_sep = (C::kRingPT < C::kSPT) && c == C::kSPT - 1;   // rope outside the ring
        const uint32_t rs = C::kRopeSlots > 0 ? g % (C::kRopeSlots > 0 ? C::kRopeSlots : 1) : 0;
        const uint32_t rph = C::kRopeSlots > 0 ? (g / (C::kRopeSlots > 0 ? C::kRopeSlots : 1)) & 1 : 0;
        const uint32_t fb = rope_sep ? smem_u32(&sh->rope_full[rs]) : smem_u32(&sh->full[slot]);
        // MXFP4: the dequantisation publishes a tile's four value chunks together, on the last
        // chunk's barrier (the first value chunk's slot is 4 (g mod 2), so that one is slot + 3).
        const bool mx_value = KV == 2 && !rope_sep;
        if ((!mx_value || c == 0) &&
            !(ok = wait_bar(mx_value ? smem_u32(&sh->full[slot + 3]) : fb, rope_sep ? rph : phase, abortf, p.status,
                            p.wait_limit_ns)))
          break;
        tc_fence_after();
        const uint64_t a = rope_sep ? ds.rope + dofs(rs * kRopeBytes) : ds.ring_k + dofs(slot * C::kSlotBytes);
        if constexpr (KV == 0) {
          const uint64_t b = ds.q + dofs(2 * c * G::kQChunk);
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f16(d, a + dofs(32 * k), b + dofs(32 * k), idq, (c | k) != 0);
          if (c < 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_f16(d, a + dofs(16384 + 32 * k), b + dofs(G::kQChunk + 32 * k), idq, 1u);
          }
        } else {
          const uint64_t b = c < 4 ? ds.q + dofs(c * G::kQChunk) : ds.q_rope;
#pragma unroll
          for (int k = 0; k < (c < 4 ? 4 : 2); ++k) mma_f8(d, a + dofs(32 * k), b + dofs(32 * k), idq, (i | k) != 0);
        }
        if (c == C::kSPT - 1)   // the rope chunk is read by QK only
          mma_commit(rope_sep ? smem_u32(&sh->rope_empty[rs]) : smem_u32(&sh->empty[slot]));
        if (!rope_sep && ++slot == G::kRing) { slot = 0; phase ^= 1; }
      }
      if (ok) mma_commit(smem_u32(&sh->s_full[g & 1]));
    }
    ++kseg;
  }
  mma_commit(smem_u32(&sh->mma_done[0]));
  wait_bar(smem_u32(&sh->mma_done[0]), 0, abortf, p.status, kDrainLimitNs, false);
}

// PV issuer `part` (0 or 1) issues the two 128-dim blocks 2*part, 2*part+1 of every tile.
template <int KV, bool PG, bool SP, int QL>
__device__ void run_mma_pv(const DecodeParams& p, SharedState* sh, const Descs& ds, uint32_t tmem, int part) {
  using C = Cfg<KV>;
  using G = Geo<KV, QL>;
  constexpr uint32_t idp = instr_desc(KV == 0 ? 1u : 0u, 1, 1, 128, G::kN);  // MN-major A (V^T) and B (P^T)
  volatile int* abortf = &sh->abort;
  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg s;
  uint32_t g = 0, slot0 = 0;                      // ring slot of chunk 0 of tile g
  int kseg = 0;
  bool ok = true;
  while (ok && it.next(p, s)) {
    const int n = s.n_hi - s.n_lo;
    if (n <= 0) continue;
    const int ntiles = (n + kBN - 1) / kBN;
    for (int t = 0; ok && t < ntiles; ++t, ++g) {
      if (!(ok = wait_bar(smem_u32(&sh->p_full[g & 1]), (g >> 1) & 1, abortf, p.status, p.wait_limit_ns))) break;
      if (t == 0 && kseg > 0 &&
          !(ok = wait_bar(smem_u32(&sh->o_free), (kseg - 1) & 1, abortf, p.status, p.wait_limit_ns)))
        break;
      tc_fence_after();
      const bool first = (t == 0);
      const uint64_t b = ds.p + dofs((G::kPBufs == 2 ? (g & 1) : 0u) * G::kPBuf);
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int m = 2 * part + mm;
        uint32_t slot = slot0 + m;
        if (slot >= G::kRing) slot -= G::kRing;
        const uint64_t a = ds.ring_mn + dofs(slot * C::kSlotBytes);
        const uint32_t d = tmem + 2 * G::kSCols + m * G::kOCols;
        // K steps of the P^T operand: 16 (bf16) or 32 (e4m3) token rows of 32 QL bytes
        if constexpr (KV == 0) {
#pragma unroll
          for (int k = 0; k < 8; ++k) mma_f16(d, a + dofs(2048 * k), b + dofs(512 * QL * k), idp, !(first && k == 0));
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f8(d, a + dofs(4096 * k), b + dofs(1024 * QL * k), idp, !(first && k == 0));
        }
        mma_commit(smem_u32(&sh->empty[slot]));
      }
      mma_commit(smem_u32(&sh->pv_done[g & 1]));   // completes once both PV issuers have committed
      slot0 += C::kRingPT;
      if (slot0 >= G::kRing) slot0 -= G::kRing;
    }
    ++kseg;
  }
  mma_commit(smem_u32(&sh->mma_done[1 + part]));
  wait_bar(smem_u32(&sh->mma_done[1 + part]), 0, abortf, p.status, kDrainLimitNs, false);
}

// ---------------------------------------------------------------- softmax / epilogue (128 threads)
// Pieces (partial results) of sequence b and their first workspace slot.
template <bool PG>
__device__ __forceinline__ int seq_pieces(const DecodeParams& p, int b, long long total, int* slot0) {
  if (p.num_splits >= 1) {
    *slot0 = b * p.num_splits;
    return p.num_splits;
  }
  const int Ge = balanced_ctas(total, p.num_ctas);
  long long r0 = p.kv_indptr[b], r1 = p.kv_indptr[b + 1];   // a merged sequence is non-empty
  int cf, cl;
  if constexpr (PG) {
    r1 = r0 * p.page_size + (r1 - r0 - 1) * p.page_size + p.last_page_len[b];
    r0 *= p.page_size;
    cf = cta_of_token<PG>(r0, total, Ge);
    cl = cta_of_token<PG>(r1 - 1, total, Ge);
  } else {
    const long long X = p.cross_rows, Tc = balanced_cost_total(total, p.batch, X);
    cf = cta_of_cost(r0 + X * b, Tc, Ge);
    cl = cta_of_cost(r1 - 1 + X * b, Tc, Ge);
  }
  *slot0 = b + cf;
  return cl - cf + 1;
}

// Log-sum-exp merge of all pieces of sequence b (run by the CTA that wrote the last piece):
// m = max_s lse_s, w_s = 2^(lse_s - m), out = sum w_s o_s / sum w_s (bf16, RNE).  Pieces
// with lse = -inf carry no weight (their partial output was never written); a row with no
// weight at all is written as 0.  One warp per head: lane l owns dims 4l + 128j (j < 4);
// weights are broadcast by shuffle and the loads of four pieces are issued together.
// Partials of other CTAs are read through L2 (ld.global.cg).
__device__ __forceinline__ uint2 pack_bf16x4(float4 v, float inv) {
  return make_uint2(static_cast<uint32_t>(f_to_bf16_bits(v.x * inv)) | (static_cast<uint32_t>(f_to_bf16_bits(v.y * inv)) << 16),
                    static_cast<uint32_t>(f_to_bf16_bits(v.z * inv)) | (static_cast<uint32_t>(f_to_bf16_bits(v.w * inv)) << 16));
}
__device__ __forceinline__ float warp_sum(float t) {
  t += __shfl_xor_sync(0xffffffffu, t, 16);
  t += __shfl_xor_sync(0xffffffffu, t, 8);
  t += __shfl_xor_sync(0xffffffffu, t, 4);
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  return t;
}

// kTwoPiece compiles the two-piece path and the skipping of empty pieces' partial loads (both
// left out of the MXFP4 kernel, whose softmax warps share the instruction cache with the
// dequantisation loop; its balanced pieces are never empty).
template <bool kTwoPiece>
__device__ void merge_pieces(const DecodeParams& p, int b, int slot0, int pieces, int ts, int nt) {
  const int warp = ts >> 5, lane = ts & 31, nw = nt >> 5;
  if (kTwoPiece && 2 * nw == kHeads && pieces == 2) {
    // Two pieces, two heads per warp: the partial outputs are loaded together with the
    // log-sum-exps (one round trip to L2; a weightless piece's unwritten partial is loaded
    // but never used).
    const int ha = warp, hb = warp + nw;
    float4 va[2][4], vb[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float4* srca = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slot0 + k) * kHeads + ha) * kDimV);
      const float4* srcb = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slot0 + k) * kHeads + hb) * kDimV);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        va[k][j] = __ldcg(srca + lane + 32 * j);
        vb[k][j] = __ldcg(srcb + lane + 32 * j);
      }
    }
    float la[2], lb[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      la[k] = __ldcg(p.part_lse + (slot0 + k) * kHeads + ha);
      lb[k] = __ldcg(p.part_lse + (slot0 + k) * kHeads + hb);
    }
    const float ma = fmaxf(la[0], la[1]), mb = fmaxf(lb[0], lb[1]);
    float ua[2], ub[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      ua[k] = la[k] == kNegInf ? 0.f : ex2(la[k] - ma);
      ub[k] = lb[k] == kNegInf ? 0.f : ex2(lb[k] - mb);
    }
    const float sa = ua[0] + ua[1], sb = ub[0] + ub[1];
    const float ia = sa > 0.f ? 1.0f / sa : 0.f, ib = sb > 0.f ? 1.0f / sb : 0.f;
    uint2* da = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * kHeads + ha) * kDimV);
    uint2* db = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * kHeads + hb) * kDimV);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (ua[k] != 0.f) {
          oa.x = fmaf(ua[k], va[k][j].x, oa.x); oa.y = fmaf(ua[k], va[k][j].y, oa.y);
          oa.z = fmaf(ua[k], va[k][j].z, oa.z); oa.w = fmaf(ua[k], va[k][j].w, oa.w);
        }
        if (ub[k] != 0.f) {
          ob.x = fmaf(ub[k], vb[k][j].x, ob.x); ob.y = fmaf(ub[k], vb[k][j].y, ob.y);
          ob.z = fmaf(ub[k], vb[k][j].z, ob.z); ob.w = fmaf(ub[k], vb[k][j].w, ob.w);
        }
      }
      da[lane + 32 * j] = pack_bf16x4(oa, ia);
      db[lane + 32 * j] = pack_bf16x4(ob, ib);
    }
    return;
  }
  if (2 * nw == kHeads && pieces <= 32) {
    // Two heads per warp, merged together: one round of log-sum-exp loads (lane s holds
    // piece s), then the partial outputs of two pieces x two heads in flight at a time.
    const int ha = warp, hb = warp + nw;
    const float la = lane < pieces ? __ldcg(p.part_lse + (slot0 + lane) * kHeads + ha) : kNegInf;
    const float lb = lane < pieces ? __ldcg(p.part_lse + (slot0 + lane) * kHeads + hb) : kNegInf;
    const float ma = warp_max(la), mb = warp_max(lb);
    const float wa = (la == kNegInf) ? 0.f : ex2(la - ma);
    const float wb = (lb == kNegInf) ? 0.f : ex2(lb - mb);
    const float sa = warp_sum(wa), sb = warp_sum(wb);
    float4 acca[4], accb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acca[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      accb[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 2
    for (int k = 0; k < pieces; ++k) {
      const float ua = __shfl_sync(0xffffffffu, wa, k), ub = __shfl_sync(0xffffffffu, wb, k);
      if (kTwoPiece && ua == 0.f && ub == 0.f) continue;   // (warp-uniform) empty piece: no partial to read
      const float4* srca = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slot0 + k) * kHeads + ha) * kDimV);
      const float4* srcb = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slot0 + k) * kHeads + hb) * kDimV);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 va = __ldcg(srca + lane + 32 * j), vb = __ldcg(srcb + lane + 32 * j);
        if (ua != 0.f) {  // a weightless piece's partial was never written: never read it into the sum
          acca[j].x = fmaf(ua, va.x, acca[j].x); acca[j].y = fmaf(ua, va.y, acca[j].y);
          acca[j].z = fmaf(ua, va.z, acca[j].z); acca[j].w = fmaf(ua, va.w, acca[j].w);
        }
        if (ub != 0.f) {
          accb[j].x = fmaf(ub, vb.x, accb[j].x); accb[j].y = fmaf(ub, vb.y, accb[j].y);
          accb[j].z = fmaf(ub, vb.z, accb[j].z); accb[j].w = fmaf(ub, vb.w, accb[j].w);
        }
      }
    }
    const float ia = sa > 0.f ? 1.0f / sa : 0.f, ib = sb > 0.f ? 1.0f / sb : 0.f;
    uint2* da = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * kHeads + ha) * kDimV);
    uint2* db = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * kHeads + hb) * kDimV);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      da[lane + 32 * j] = pack_bf16x4(acca[j], ia);
      db[lane + 32 * j] = pack_bf16x4(accb[j], ib);
    }
    return;
  }
  for (int h = warp; h < kHeads; h += nw) {
    float m = kNegInf;
    for (int s = lane; s < pieces; s += 32) m = fmaxf(m, __ldcg(p.part_lse + (slot0 + s) * kHeads + h));
    m = warp_max(m);
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    float ws = 0.f;
    if (m != kNegInf) {
      for (int s0 = 0; s0 < pieces; s0 += 32) {
        const int cnt = min(32, pieces - s0);
        const float l = lane < cnt ? __ldcg(p.part_lse + (slot0 + s0 + lane) * kHeads + h) : kNegInf;
        const float myw = (l == kNegInf) ? 0.f : ex2(l - m);
        float t = myw;
        t += __shfl_xor_sync(0xffffffffu, t, 16);
        t += __shfl_xor_sync(0xffffffffu, t, 8);
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        ws += t;
#pragma unroll 4
        for (int k = 0; k < cnt; ++k) {
          const float w = __shfl_sync(0xffffffffu, myw, k);
          if (kTwoPiece && w == 0.f) continue;   // (warp-uniform) empty piece: no partial to read
          const float4* src =
              reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slot0 + s0 + k) * kHeads + h) * kDimV);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = __ldcg(src + lane + 32 * j);
            if (w != 0.f) {  // a weightless piece's partial was never written: never read it into the sum
              acc[j].x = fmaf(w, v.x, acc[j].x);
              acc[j].y = fmaf(w, v.y, acc[j].y);
              acc[j].z = fmaf(w, v.z, acc[j].z);
              acc[j].w = fmaf(w, v.w, acc[j].w);
            }
          }
        }
      }
    }
    const float inv = ws > 0.f ? 1.0f / ws : 0.f;
    uint2* dst = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(b) * kHeads + h) * kDimV);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = static_cast<uint32_t>(f_to_bf16_bits(acc[j].x * inv)) |
                          (static_cast<uint32_t>(f_to_bf16_bits(acc[j].y * inv)) << 16);
      const uint32_t hi = static_cast<uint32_t>(f_to_bf16_bits(acc[j].z * inv)) |
                          (static_cast<uint32_t>(f_to_bf16_bits(acc[j].w * inv)) << 16);
      dst[lane + 32 * j] = make_uint2(lo, hi);
    }
  }
}

// After this CTA wrote its piece of sequence s.b: count the piece; the CTA whose piece
// completes the count merges all pieces and re-arms the counter for the next call.
// Reached by all `nt` softmax threads.
template <int KV, bool PG>
__device__ void finish_piece(const DecodeParams& p, SharedState* sh, const Seg& s, int ts, int nt) {
  __threadfence();
  bar_sync(1, nt);
  if (ts == 0) {
    int slot0 = 0;
    const int pieces = seq_pieces<PG>(p, s.b, sh->seg_total, &slot0);
    const int old = atomicAdd(p.seq_count + s.b, 1);
    const bool last = (old == pieces - 1);
    if (last) {
      p.seq_count[s.b] = 0;
      fence_acq_rel_gpu();   // the other pieces' partials (released by their fence + count)
    }
    sh->merge_slot0 = slot0;
    sh->merge_pieces = last ? pieces : 0;
  }
  bar_sync(1, nt);
  const int pieces = sh->merge_pieces;
  if (pieces > 0) merge_pieces<KV != 2>(p, s.b, sh->merge_slot0, pieces, ts, nt);
}

template <int KV>
__device__ void write_empty_result(const DecodeParams& p, const Seg& s, int ts) {
  if (s.direct) {
    uint32_t* o = reinterpret_cast<uint32_t*>(p.out + static_cast<size_t>(s.b) * kHeads * kDimV);
    for (int i = ts; i < kHeads * kDimV / 2; i += Cfg<KV>::kSoftWarps * 32) o[i] = 0u;
  } else if (ts < kHeads) {
    p.part_lse[s.slot * kHeads + ts] = kNegInf;
  }
}

// Softmax / epilogue warps.  Thread = one token of the tile (= one TMEM lane) for H heads:
// kSoftWarps = 8 puts two warps on each TMEM lane quarter, each owning 8 heads (halving the
// per-tile latency of this stage); kSoftWarps = 4 gives each thread all 16 heads.  The two
// head groups never share a named barrier on a path the other may skip: every named
// barrier below is reached by all softmax threads once per tile (or once per segment).
// QL = 2 (fused multi-token instances): the thread owns its H heads for both query tokens of
// the segment, K = QL H columns; column k is token k / H, head h0 + k % H.  Token j of a
// segment of `rows` query rows sees the first n_total - (rows - 1 - j) cached tokens (the
// causal mask of the multi-token interface); a token with no visible row in the segment
// gets P = 0 and a piece with log-sum-exp -inf (or a zero output row).
template <int KV, bool PG, int QL>
__device__ void run_softmax(const DecodeParams& p, SharedState* sh, uint8_t* qs, uint8_t* ps, uint32_t tmem) {
  using C = Cfg<KV>;
  using G = Geo<KV, QL>;
  constexpr int NW = C::kSoftWarps;
  constexpr int NT = NW * 32;
  constexpr int H = 64 / NW;                               // heads per thread: 16 or 8
  constexpr int K = QL * H;                                // columns per thread
  volatile int* abortf = &sh->abort;
  const int ts = threadIdx.x - 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int hg = (ts >> 5) >> 2;                           // head group (0 when H = 16)
  const int h0 = hg * H;
  const int row = quarter * 32 + lane;                     // token row of the tile = TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  float kv_scale = 1.0f;
  if constexpr (KV == 1) kv_scale = __ldg(reinterpret_cast<const float*>(p.kv_scale));
  const float xscale = p.logit_scale_log2 * kv_scale;    // raw dot product -> log2-domain logit
  // Column k -> index 16 j + h of the per-(token, head) shared arrays.
  auto cidx = [&](int k) { return 16 * (k / H) + h0 + (k % H); };

  SegIter<PG> it;
  it.init(p, blockIdx.x, sh);
  Seg cur, nxt;
  bool has_cur = it.next(p, cur);
  // Stage q of the first non-empty segment (the iterator may first yield empty ones).
  auto stage_next_nonempty = [&](const SegIter<PG>& from, const Seg* first) {
    Seg sn;
    bool found = false;
    if (first != nullptr && first->n_hi > first->n_lo) { sn = *first; found = true; }
    SegIter<PG> look = from;
    while (!found && look.next(p, sn)) found = sn.n_hi > sn.n_lo;
    if (found && ts < 128 * QL) {
      if constexpr (KV == 0) stage_q_bf16<QL>(p, sn.b, sn.rows, qs, ts);
      else stage_q_fp8<QL>(p, sn.b, sn.rows, qs, sh->qscale, ts);
      fence_proxy_async_smem();
      warp_arrive(smem_u32(&sh->q_ready));
    }
  };
  // The single-row segment of query token j of `s` (output row, partial slot).
  auto token_seg = [&](const Seg& s, int j) {
    Seg r = s;
    r.b = s.b + j;
    r.slot = s.slot + j * p.num_splits;
    return r;
  };
  if (has_cur) stage_next_nonempty(it, &cur);
  bar_sync(1, NT);  // qscale visible to all softmax threads
  uint32_t g = 0;
  bool ok = true;
  while (ok && has_cur) {
    const int n = cur.n_hi - cur.n_lo;
    if (n <= 0) {
      for (int j = 0; j < cur.rows; ++j) {
        const Seg sj = token_seg(cur, j);
        write_empty_result<KV>(p, sj, ts);
        if (!sj.direct) finish_piece<KV, PG>(p, sh, sj, ts, NT);
      }
      has_cur = it.next(p, cur);
      continue;
    }
    // Per-column logit multiplier (QL = 2: read from shared memory where it is used, which
    // keeps 16 registers free in these instances).
    float qx[QL == 1 ? K : 1];
    if constexpr (QL == 1) {
#pragma unroll
      for (int k = 0; k < K; ++k) qx[k] = (KV == 0) ? xscale : sh->qscale[cidx(k)] * xscale;
    }
    const int ntiles = (n + kBN - 1) / kBN;
    float mref[K], lpart[K];
    bool has_nxt = false;
    for (int t = 0; t < ntiles; ++t) {
      const Window w = tile_window<KV, PG>(p, cur, t);
      bool okw = wait_bar(smem_u32(&sh->s_full[g & 1]), (g >> 1) & 1, abortf, p.status, p.wait_limit_ns);
      okw = __all_sync(0xffffffffu, okw);
      tc_fence_after();
      uint32_t rh[QL][H], rl[QL][H];
      if (okw) {
#pragma unroll
        for (int j = 0; j < QL; ++j) {
          const uint32_t ta = tmem + lane_base + (g & 1) * G::kSCols + j * G::kTokCols + h0;
          tmem_ld<H>(ta, rh[j]);
          if constexpr (KV != 0) tmem_ld<H>(ta + 16, rl[j]);
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      warp_arrive(smem_u32(&sh->s_free[g & 1]));
      const bool valid = okw && row >= w.shift && row < w.shift + w.cnt;
      bool vtok[QL];
      vtok[0] = valid;
      if constexpr (QL == 2) {
        // token index of this row in the sequence (paged windows start at the tile's token)
        const int tok = cur.n_lo + t * kBN + row;
#pragma unroll
        for (int j = 0; j < QL; ++j) vtok[j] = valid && j < cur.rows && tok < cur.n_total - (cur.rows - 1 - j);
      }
      // MXFP4 rows carry a power-of-two factor 2^eadd (eadd = e_row - 127): logits are
      // scaled by it, P is weighted by it (w = x + eadd) and the softmax sum is not.
      float eadd = 0.f, rowf = 1.f;
      if constexpr (KV == 2) {
        bool oke = wait_bar(smem_u32(&sh->etok_full[g & 3]), (g >> 2) & 1, abortf, p.status, p.wait_limit_ns);
        okw = okw && oke;
        const int e = sh->etok[g & 3][row];
        eadd = static_cast<float>(e - 127);
        rowf = pow2i(e - 127);
      }
      // One pass per query token: its logits, the row maximum across the tile (warp max and
      // the cross-warp exchange), the lazy rescale of its O columns, its P.  (QL = 2: the
      // two passes keep half the per-column state live at a time.)
      bool okt = okw;
#pragma unroll
      for (int j = 0; j < QL; ++j) {
        float x[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const int k = j * H + h;
          float sdot;
          if constexpr (KV == 0) sdot = __uint_as_float(rh[j][h]);
          else sdot = fmaf(__uint_as_float(rl[j][h]), 0.0625f, __uint_as_float(rh[j][h])) * rowf;
          float qk;
          if constexpr (QL == 1) qk = qx[k];
          else qk = (KV == 0) ? xscale : sh->qscale[cidx(k)] * xscale;
          x[h] = vtok[j] ? fmaf(sdot, qk, eadd) : kNegInf;
        }
        float* red = &sh->red[g & 1][quarter][16 * j + h0];
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const float m = warp_max(x[h]);
          if (lane == 0) red[h] = m;
        }
        okt = bar_and(1, NT, okt);
        if (!okt) break;
        float M[H];
#pragma unroll
        for (int h4 = 0; h4 < H; h4 += 4) {
          const int c0 = 16 * j + h0 + h4;
          const float4 a = *reinterpret_cast<const float4*>(&sh->red[g & 1][0][c0]);
          const float4 b = *reinterpret_cast<const float4*>(&sh->red[g & 1][1][c0]);
          const float4 c = *reinterpret_cast<const float4*>(&sh->red[g & 1][2][c0]);
          const float4 d = *reinterpret_cast<const float4*>(&sh->red[g & 1][3][c0]);
          M[h4 + 0] = fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x));
          M[h4 + 1] = fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y));
          M[h4 + 2] = fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z));
          M[h4 + 3] = fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w));
        }
        float* mr = &mref[j * H];
        float* lp = &lpart[j * H];
        bool need = false;
        if (t == 0) {
#pragma unroll
          for (int h = 0; h < H; ++h) { mr[h] = M[h]; lp[h] = 0.f; }
        } else {
#pragma unroll
          for (int h = 0; h < H; ++h) need |= (M[h] > mr[h] + C::kTau);
        }
        if (need) {  // lazy rescale of this head group's O^T columns of token j (uniform within the group)
          float alpha[H];
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const float nm = fmaxf(mr[h], M[h]);
            alpha[h] = ex2(mr[h] - nm);
            mr[h] = nm;
            lp[h] *= alpha[h];
          }
          const uint32_t gp = g - 1;
          bool ok2 = wait_bar(smem_u32(&sh->pv_done[gp & 1]), (gp >> 1) & 1, abortf, p.status, p.wait_limit_ns);
          ok2 = __all_sync(0xffffffffu, ok2);
          if (ok2) {
            tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
#pragma unroll
              for (int part = 0; part < (KV == 0 ? 1 : 2); ++part) {
                const uint32_t ta =
                    tmem + lane_base + 2 * G::kSCols + m * G::kOCols + j * G::kTokCols + part * 16 + h0;
                uint32_t v[H];
                tmem_ld<H>(ta, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < H; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha[i]);
                tmem_st<H>(ta, v);
              }
            }
            tmem_wait_st();
          }
          // A failed wait has set the abort flag and the status word.  The warp carries on: the
          // softmax warps learn of the abort at their next waits and leave together at the next
          // named barrier (a warp leaving alone would strand the others there).
        }
        // P = 2^(w - mref) <= 2^kTau (QL = 2: a column with no visible row yet has mref = -inf)
        float P[H];
#pragma unroll
        for (int h = 0; h < H; ++h) P[h] = ex2(x[h] - ((QL == 2 && mr[h] == kNegInf) ? 0.f : mr[h]));
        // The P^T buffer was last read by the PV MMAs of tile g - 2 (two buffers) or g - 1 (one).
        if constexpr (G::kPBufs == 2) {
          if (j == 0 && g >= 2)
            wait_bar(smem_u32(&sh->pv_done[g & 1]), ((g >> 1) & 1) ^ 1, abortf, p.status, p.wait_limit_ns);
        } else {
          if (j == 0 && g >= 1)
            wait_bar(smem_u32(&sh->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abortf, p.status, p.wait_limit_ns);
        }
        // P^T row of this token: 32 QL bytes (per query token: 16 heads of hi then of lo e4m3,
        // or 16 bf16); swizzled in 16-byte chunks, 32-byte (QL = 1) or 64-byte (QL = 2) pattern.
        uint8_t* prow = ps + (G::kPBufs == 2 ? (g & 1) : 0u) * G::kPBuf + row * 32 * QL;
        const int sw = QL == 1 ? (row >> 2) & 1 : (row >> 1) & 3;
        if constexpr (KV == 0) {
          uint32_t wv[H / 2];
#pragma unroll
          for (int i = 0; i < H / 2; ++i) {
            const uint16_t b0 = f_to_bf16_bits(P[2 * i]), b1 = f_to_bf16_bits(P[2 * i + 1]);
            lp[2 * i] += bf16_bits_to_f(b0);
            lp[2 * i + 1] += bf16_bits_to_f(b1);
            wv[i] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
          }
          // heads [h0, h0 + H) of token j are 16-byte chunk(s) 2 j + h0/8 .. of the row
#pragma unroll
          for (int c = 0; c < H / 8; ++c)
            *reinterpret_cast<uint4*>(prow + (((2 * j + h0 / 8 + c) ^ sw) << 4)) =
                make_uint4(wv[4 * c], wv[4 * c + 1], wv[4 * c + 2], wv[4 * c + 3]);
        } else {
          // Softmax sum: fp8 caches add the e4m3-rounded P (the values the PV MMAs weight V
          // with).  MXFP4 rows add the fp32 P * 2^-eadd: a row of small magnitude (eadd << 0)
          // can carry a large softmax weight with a PV weight too small for e4m3.
          const float einv = pow2i(-static_cast<int>(eadd) - 4);   // 2^-eadd / 16
          const float escale = pow2i(-static_cast<int>(eadd));      // 2^-eadd
          uint32_t hw[H / 4], lw[H / 4];
#pragma unroll
          for (int i = 0; i < H / 4; ++i) {
            uint32_t a = 0, b = 0;
#pragma unroll
            for (int kk = 0; kk < 4; kk += 2) {
              const int h = 4 * i + kk;
              const float y0 = P[h] * 16.f, y1 = P[h + 1] * 16.f;
              const uint32_t hp = pack_e4m3x2(y0, y1);
              const float2 hd = unpack_e4m3x2(hp);
              const uint32_t lpk = pack_e4m3x2((y0 - hd.x) * 16.f, (y1 - hd.y) * 16.f);
              if constexpr (KV == 2) {
                lp[h] = fmaf(P[h], escale, lp[h]);
                lp[h + 1] = fmaf(P[h + 1], escale, lp[h + 1]);
              } else {
                const float2 ld = unpack_e4m3x2(lpk);
                lp[h] += fmaf(ld.x, 0.0625f, hd.x) * einv;
                lp[h + 1] += fmaf(ld.y, 0.0625f, hd.y) * einv;
              }
              a |= hp << (8 * kk);
              b |= lpk << (8 * kk);
            }
            hw[i] = a;
            lw[i] = b;
          }
          if constexpr (H == 16) {
            *reinterpret_cast<uint4*>(prow + (((2 * j) ^ sw) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(prow + (((2 * j + 1) ^ sw) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          } else {
            *reinterpret_cast<uint2*>(prow + (((2 * j) ^ sw) << 4) + h0) = make_uint2(hw[0], hw[1]);
            *reinterpret_cast<uint2*>(prow + (((2 * j + 1) ^ sw) << 4) + h0) = make_uint2(lw[0], lw[1]);
          }
        }
      }
      ok = okt;
      if (!ok) break;
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(smem_u32(&sh->p_full[g & 1]));
      ++g;
      if (t == ntiles - 1) {
        // All QK MMAs of this segment are complete (s_full of its last tile was observed):
        // the q buffer can take the next segment's queries.
        has_nxt = it.next(p, nxt);
        if (has_nxt) stage_next_nonempty(it, &nxt);
      }
    }
    if (!ok) break;
    // ---- epilogue: O = O^T / l, written directly (bf16) or as a partial (fp32 + lse)
    const uint32_t gl = g - 1;
    bool ok4 = wait_bar(smem_u32(&sh->pv_done[gl & 1]), (gl >> 1) & 1, abortf, p.status, p.wait_limit_ns);
    ok4 = __all_sync(0xffffffffu, ok4);
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float v = lpart[k];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) sh->lsum[quarter][cidx(k)] = v;
    }
    ok = bar_and(1, NT, ok4);
    if (!ok) break;
    float inv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int c = cidx(k), j = k / H;
      const float l = sh->lsum[0][c] + sh->lsum[1][c] + sh->lsum[2][c] + sh->lsum[3][c];
      inv[k] = __fdividef(KV == 0 ? 1.0f : kv_scale * 0.0625f, l);
      if constexpr (QL == 2) inv[k] = l > 0.f ? inv[k] : 0.f;   // a token with no visible row: zeros
      if (!cur.direct && quarter == 0 && lane == 0 && j < cur.rows)
        p.part_lse[(cur.slot + j * p.num_splits) * kHeads + (k % H) + h0] = mref[k] + lg2(l);
    }
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int j = 0; j < QL; ++j) {
        const uint32_t ta = tmem + lane_base + 2 * G::kSCols + m * G::kOCols + j * G::kTokCols + h0;
        uint32_t vh[H], vl[H];
        tmem_ld<H>(ta, vh);
        if constexpr (KV != 0) tmem_ld<H>(ta + 16, vl);
        tmem_wait_ld();
        if (j >= cur.rows) continue;
        const int d = 128 * m + row;
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float o = __uint_as_float(vh[h]);
          if constexpr (KV != 0) o = fmaf(__uint_as_float(vl[h]), 0.0625f, o);
          o *= inv[j * H + h];
          if (cur.direct)
            p.out[(static_cast<size_t>(cur.b + j) * kHeads + h0 + h) * kDimV + d] = f_to_bf16_bits(o);
          else
            p.part_o[(static_cast<size_t>(cur.slot + j * p.num_splits) * kHeads + h0 + h) * kDimV + d] = o;
        }
      }
    }
    tc_fence_before();
    warp_arrive(smem_u32(&sh->o_free));
    if (!cur.direct) {
      for (int j = 0; j < cur.rows; ++j) finish_piece<KV, PG>(p, sh, token_seg(cur, j), ts, NT);
    }
    cur = nxt;
    has_cur = has_nxt;
  }
}

// ---------------------------------------------------------------- the kernel
// PG: paged cache.  SP: pages of 1, 2 or 4 rows (four-row gathers; MXFP4 slabs: cp.async).
// QL: query tokens decoded together (2: the fused multi-token instances).
template <int KV, bool PG, bool SP, int QL>
__global__ void __launch_bounds__(Cfg<KV>::kThreads, 1) mla_split_kernel(const __grid_constant__ DecodeParams p) {
  using C = Cfg<KV>;
  using G = Geo<KV, QL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = base;
  uint8_t* rope = ring + G::kRing * C::kSlotBytes;
  uint8_t* qs = rope + rope_bytes<KV>();
  uint8_t* ps = qs + G::kQBytes;
  uint8_t* slabs = ps + G::kPBufs * G::kPBuf;        // MXFP4 packed-row staging
  SharedState* sh = reinterpret_cast<SharedState*>(slabs + raw_bytes<KV>());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::kRing; ++i) {
      // MXFP4: one arrival per dequant warp (on the last value slot of each tile); otherwise
      // the producer's expected-bytes arrival
      mbar_init(smem_u32(&sh->full[i]), KV == 2 ? C::kDeqWarps : 1);
      mbar_init(smem_u32(&sh->empty[i]), 1);
    }
    if (KV == 2) {
      for (int i = 0; i < kSlabs; ++i) {
        mbar_init(smem_u32(&sh->slab_full[i]), SP ? 32 : 1);   // pages of 1-4 rows: one cp.async arrival per producer lane
        mbar_init(smem_u32(&sh->slab_empty[i]), C::kDeqWarps);   // one arrival per dequant warp
      }
      for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&sh->etok_full[i]), C::kDeqWarps);

    }
    // softmax-side barriers count warps (one arrival per warp)
    mbar_init(smem_u32(&sh->q_ready), 4 * QL);  // four softmax warps per query token stage q
    for (int i = 0; i < C::kRopeSlots; ++i) {
      mbar_init(smem_u32(&sh->rope_full[i]), KV == 2 ? C::kDeqWarps : 1);   // MXFP4: per dequant warp
      mbar_init(smem_u32(&sh->rope_empty[i]), 1);                          // QK commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->s_free[i]), C::kSoftWarps);
      mbar_init(smem_u32(&sh->p_full[i]), C::kSoftWarps);
      mbar_init(smem_u32(&sh->pv_done[i]), 2);   // one commit from each PV issuer
    }
    mbar_init(smem_u32(&sh->o_free), C::kSoftWarps);
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&sh->mma_done[i]), 1);
    mbar_init(smem_u32(&sh->never), 1);
    sh->abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), G::kTmemCols);
    tmem_relinquish();
  }
  // Programmatic dependent launch: the set-up above (barrier init, TMEM allocation) may run
  // while the previous kernel in the stream finishes; every global memory access of this
  // kernel comes after this wait.  The next kernel may begin its own set-up as soon as
  // every CTA of this one is running.
  grid_dep_launch_dependents();
  grid_dep_wait();
  if (warp == 0 && p.num_splits < 1) {
    // Balanced mode: this CTA's position range [lo, hi) and its first sequence b0, the first
    // b with kv_indptr[b+1] >= lo (paged: kv_indptr[b+1] * P >= lo): empty sequences sitting
    // at lo are this CTA's too.
    const long long total = static_cast<long long>(p.kv_indptr[p.batch]) * (PG ? p.page_size : 1);
    const int Ge = balanced_ctas(total, p.num_ctas);
    const int c = static_cast<int>(blockIdx.x);
    int b0 = p.batch;
    long long lo = total, hi = total;
    if (c < Ge) {
      if constexpr (PG) {   // row cuts rounded to whole tiles (cta_lo)
        lo = cta_lo<PG>(c, total, Ge);
        hi = cta_lo<PG>(c + 1, total, Ge);
        b0 = warp_first_seq(p.kv_indptr, p.batch, (lo + p.page_size - 1) / p.page_size - 1);
      } else {              // cost cuts (balanced_cost_total)
        const long long X = p.cross_rows, Tc = balanced_cost_total(total, p.batch, X);
        const long long clo = static_cast<long long>(c) * Tc / Ge, chi = static_cast<long long>(c + 1) * Tc / Ge;
        int blo, bhi;
        warp_first_seq_cost2(p.kv_indptr, p.batch, X, clo, chi, &blo, &bhi);
        if (blo < p.batch) lo = min(clo - X * blo, static_cast<long long>(p.kv_indptr[blo + 1]));
        if (c + 1 < Ge && bhi < p.batch) hi = min(chi - X * bhi, static_cast<long long>(p.kv_indptr[bhi + 1]));
        b0 = blo;
        while (b0 > 0 && p.kv_indptr[b0] >= lo) --b0;
      }
    }
    if (lane == 0) { sh->seg_total = total; sh->seg_b0 = b0; sh->seg_lo = lo; sh->seg_hi = hi; }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  // Role dispatch by warpgroup: issuers (warps 0-3) | softmax | dequant (MXFP4).  Each
  // register-budget change sits at the top of its warpgroup's branch, so that the role's
  // code is compiled for that budget.
  if (warp < 4) {
    if constexpr (G::kSplitRegs) regs_dec<G::kRegsIssue>();
    if (warp == 0) {
      if (PG || lane == 0) {   // paged: the whole warp (one lane per page)
        if constexpr (SP) run_producer_sp<KV, QL>(p, sh, ring, rope, slabs, lane);
        else if constexpr (KV == 2) run_producer_mx<PG>(p, sh, slabs, lane);
        else run_producer<KV, PG, QL>(p, sh, ring, rope, lane);
      }
    } else if (warp == 1) {
      if (lane == 0) run_mma_qk<KV, PG, SP, QL>(p, sh, make_descs<QL>(ring, rope, qs, ps), tmem);
    } else {
      if (lane == 0) run_mma_pv<KV, PG, SP, QL>(p, sh, make_descs<QL>(ring, rope, qs, ps), tmem, warp - 2);
    }
    __syncwarp();
  } else if (warp < 4 + C::kSoftWarps) {
    if constexpr (G::kSplitRegs) regs_inc<G::kRegsSoft>();
    run_softmax<KV, PG, QL>(p, sh, qs, ps, tmem);
  } else {
    if constexpr (KV == 2) {
      regs_dec<C::kRegsDeq>();
      run_dequant<PG>(p, sh, ring, rope, slabs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

constexpr int kMaxDevices = 64;

// Per-device, once: the kernel's dynamic shared-memory limit (a per-function attribute
// that each device context keeps) and, for the instances with a register split, its check.  Thread-safe;
// the outcome of the first attempt on a device is kept.
template <int KV, bool PG, bool SP, int QL>
cudaError_t configure_once(int dev) {
  static std::once_flag once[kMaxDevices];
  static cudaError_t result[kMaxDevices];
  std::call_once(once[dev], [dev] {
    cudaError_t e = cudaFuncSetAttribute(mla_split_kernel<KV, PG, SP, QL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<KV, QL>()));
    if (e == cudaSuccess && Geo<KV, QL>::kSplitRegs) {
      // The register split's increases only complete if the CTA launched with at least the
      // registers the split hands out: refuse to launch otherwise.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, mla_split_kernel<KV, PG, SP, QL>);
      if (e == cudaSuccess && fa.numRegs * Cfg<KV>::kThreads < Geo<KV, QL>::kRegsNeeded)
        e = cudaErrorInvalidConfiguration;
    }
    result[dev] = e;
  });
  return result[dev];
}

template <int KV, bool PG, bool SP, int QL = 1>
cudaError_t launch_split_t(const DecodeParams& p, int grid, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if ((e = configure_once<KV, PG, SP, QL>(dev)) != cudaSuccess) return e;
  // Launched with programmatic stream serialisation: the kernel's set-up overlaps the tail
  // of the previous kernel in the stream (see grid_dep_wait in the kernel).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Cfg<KV>::kThreads);
  cfg.dynamicSmemBytes = smem_bytes<KV, QL>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_split_kernel<KV, PG, SP, QL>, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

}  // namespace

cudaError_t launch_split(int kv_dtype, const DecodeParams& p, int grid, cudaStream_t stream) {
  if (kv_dtype == 0) return launch_split_t<0, false, false>(p, grid, stream);
  if (kv_dtype == 1) return launch_split_t<1, false, false>(p, grid, stream);
  if (kv_dtype == 2) return launch_split_t<2, false, false>(p, grid, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_split_paged(int kv_dtype, const DecodeParams& p, int grid, cudaStream_t stream) {
  if (p.pair_rows) {              // several query tokens per sequence, two decoded together
    const bool sp = p.page_size < kMinPage;
    if (kv_dtype == 0) return sp ? launch_split_t<0, true, true, 2>(p, grid, stream) : launch_split_t<0, true, false, 2>(p, grid, stream);
    if (kv_dtype == 1) return sp ? launch_split_t<1, true, true, 2>(p, grid, stream) : launch_split_t<1, true, false, 2>(p, grid, stream);
    return cudaErrorNotSupported;
  }
  if (p.page_size < kMinPage) {   // pages of 1, 2 or 4 rows (run_producer_sp)
    if (kv_dtype == 0) return launch_split_t<0, true, true>(p, grid, stream);
    if (kv_dtype == 1) return launch_split_t<1, true, true>(p, grid, stream);
    if (kv_dtype == 2) return launch_split_t<2, true, true>(p, grid, stream);
    return cudaErrorNotSupported;
  }
  if (kv_dtype == 0) return launch_split_t<0, true, false>(p, grid, stream);
  if (kv_dtype == 1) return launch_split_t<1, true, false>(p, grid, stream);
  if (kv_dtype == 2) return launch_split_t<2, true, false>(p, grid, stream);
  return cudaErrorNotSupported;
}


}  // namespace mla
