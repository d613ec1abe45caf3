// sample.cu -- fused bitmask + temperature + top-k ∩ top-p ∩ min-p + Gumbel-max
// sampler (Kernel Hub "logits-processor", Ops "sample" and "How it works";
// unsatisfiable rows as in TensorRT-Edge-LLM "Guided Decoder").
//
// GB300 design: two kernels per call.
//
// The stream kernel makes the one pass over HBM, through the Tensor Memory
// Accelerator, in a persistent grid of three CTAs per SM.  Every row is cut into
// tiles of equal length (8-64 KB of logits) and the CTAs take the tiles of all
// rows round-robin, so the work per SM is even whatever the batch size and
// vocabulary.  A CTA streams its tiles through a ring of three 14 KB
// shared-memory stages: a producer warp keeps bulk copies (cp.async.bulk, with
// the stage's bitmask words) in flight on mbarriers, and seven consumer warps
// take each landed stage from shared memory, four 16-byte vectors per thread.
// Per tile:
//   * candidate max with its lowest index, the candidate count and, for top-p
//     rows, an online softmax sum;
//   * filtered rows: every candidate within a window below the tile's running
//     maximum is appended to a shared-memory compaction buffer.  The window is
//     exactly the min-p bound when min-p is on (max + T ln min_p); otherwise a
//     number of temperature units growing with ln(1 / (1 - top_p)) for top-p and
//     a fixed number of logits for top-k.  No tile maximum exceeds the row
//     maximum, so the tiles' buffers together hold every candidate in
//     [row max - window, row max];
//   * rows without filters draw Gumbel-max directly (no threshold needed),
//     skipping any token whose best possible score is below the running best.
// The tile's summary and buffer go to a caller-provided device workspace with
// plain stores: the buffer to the tile's own slot, or -- when longer than a
// slot -- to a shared pool.  Nothing in the stream waits on another CTA.
//
// The finish kernel (one CTA per row, launched as a programmatic dependent of
// the stream kernel so that its launch overlaps the stream) merges the row's
// tile summaries: no candidate -> -1; greedy -> argmax; unfiltered -> the best
// score's token.  Filtered rows find the keep-threshold max(t_k, t_p, t_m) as
// the largest logit at which "count >= k" or "mass >= top_p S" first holds
// (counts for top-k, 2^-40 fixed-point softmax mass for top-p): by counting when
// few candidates are staged, else by an MSD radix select over the
// order-preserving key of the logit.  The selection reads the tiles' buffers (L2
// resident), counting only the region where they are complete; if the threshold
// is not there (or a buffer overflowed) the CTA reads the row again: a strided
// sample bounds the threshold so that one pass can stage every candidate above
// it, else a window search or the radix passes run over the re-read row.  The
// draw is Gumbel-max over the kept set with Philox4x32-10 noise keyed by
// (seed, row, offset).
// Masses are integers, so every sum over tiles or warps is exact and
// order-independent; softmax sums are merged in a fixed order.  Results are
// deterministic in (seed, offset).
#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace lp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kConsumerWarps = kWarps - 1;  // stream kernel: the last warp is the producer
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kRing = 3;                 // stages in flight per CTA
constexpr int kPieceBytes = 14336;       // bytes of logits per stage: four vectors per consumer
constexpr int kPieceWords = kPieceBytes / 2 / 32 + 2;  // bitmask words a stage can need
constexpr int kMaskSlot = (16 + 4 * kPieceWords + 15) / 16 * 16;
constexpr int kPerPiece = kPieceBytes / 16 / kConsumers;  // vectors of a piece per consumer
static_assert(kPerPiece * 16 * kConsumers == kPieceBytes, "a piece is whole vectors per consumer");
constexpr int kTileBytesMax = 65536;     // longest tile
constexpr int kTileBytesMin = 8192;      // shortest tile (small batches)
constexpr int64_t kTileTarget = 1024;    // tiles per launch that shorter tiles aim for
constexpr int kCompactBytes = 24576;     // shared memory of the compaction buffers
constexpr int kSlotCap = 256;            // entries a tile keeps in its own workspace slot
constexpr int kStage = 4096;             // buffered entries a finishing CTA stages
constexpr int kWinBins = 2048;           // bins of the fallback's window search
static_assert(kWinBins % kThreads == 0, "whole bins per thread");
constexpr int kMetaCap = 1024;           // tiles per row whose buffer starts it stages
constexpr int kFinishSmem = kStage * 8 + (kMetaCap + 1) * 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWindowK = 6.f;          // top-k window, in logits
constexpr int kSmem = kRing * kPieceBytes + kRing * kMaskSlot + kCompactBytes;
// A compaction entry is the logit's own bits (4 or 2 bytes) and the token's
// offset into the tile (2 bytes); the buffer is double-buffered by tile parity.
static_assert(kTileBytesMax / 2 <= 65536, "tile offsets fit in 16 bits");
template <int DT>
struct Compact {
  using Val = std::conditional_t<DT == LP_F32, float, uint16_t>;
  static constexpr int kCapT = kCompactBytes / 2 / int(sizeof(Val) + 2);  // entries per tile
  __device__ static __forceinline__ Val pack(const uint4& v, int e) {
    if constexpr (DT == LP_F32) {
      return Elt<DT>::get(v, e);
    } else {
      return uint16_t(word_of(v, e >> 1) >> (16 * (e & 1)));
    }
  }
  __device__ static __forceinline__ float unpack(Val x) {
    if constexpr (DT == LP_F32) {
      return x;
    } else if constexpr (DT == LP_BF16) {
      return __uint_as_float(uint32_t(x) << 16);
    } else {
      return Elt<LP_F16>::half_bits_to_float(x);
    }
  }
};
constexpr uint32_t kMaxWaitTries = 1u << 22;
constexpr int kTestWaits = 8;            // non-blocking tests before an mbarrier wait suspends
constexpr int64_t kMaxTileSums = int64_t(1) << 20;  // tiles per launch
constexpr int64_t kMaxRowsPerLaunch = 16384;
constexpr int64_t kPoolPerRow = 8192;    // pooled compaction entries per row
constexpr int64_t kPoolMin = int64_t(1) << 16;
constexpr int64_t kPoolMax = int64_t(1) << 24;
constexpr uint32_t kTileOverflow = 1u << 30;
// row modes of the stream kernel's piece loop
constexpr int kModeGreedy = 0;      // max and argmax only
constexpr int kModeTopP = 1;        // + softmax sum and the compaction buffer
constexpr int kModeFilter = 2;      // + the compaction buffer (top-k, min-p)
constexpr int kModeUnfiltered = 3;  // + Gumbel-max in the stream
constexpr uint32_t kTileError = 1u << 31;

// ------------------------------------------------------------ workspace

struct WsHeader {       // one per workspace
  unsigned pool_used;   // pool entries handed out by the running stream kernel
  unsigned pad[63];
};
struct TileSum {  // one per tile of a launch
  float max;
  int arg;    // lowest index of max
  float sum;  // softmax sum relative to max (top-p rows)
  int ncand;  // candidate bits seen (-inf logits included)
  float best;
  int best_v;     // unfiltered rows: best Gumbel score and its token
  unsigned off;   // buffer longer than a slot: pool entries [off, off + n)
  unsigned nf;    // n | kTileOverflow | kTileError
};

struct SampleArgs {
  const char* logits;
  int64_t stride_bytes;
  int V;
  int row0;   // first row of this launch
  int nrows;  // rows in this launch
  int tpr;    // tiles per row
  int chunk;  // tokens per tile (a multiple of 32)
  int64_t ntiles;
  const uint32_t* bitmask;  // nullptr: no row is masked
  int64_t bm_stride;
  int64_t bm_rows;
  const int32_t* indices;   // nullptr: every row masked (when bitmask != nullptr)
  int n_indices;
  const float* temp;
  float temp_s;
  const int32_t* topk;
  int32_t topk_s;
  const float* topp;
  float topp_s;
  const float* minp;
  float minp_s;
  uint64_t seed, offset;
  int rps;                // rows per slot: row b takes the parameters at b / rps
  const uint64_t* seeds;  // [rows] per-row Philox keys, or nullptr for seed
  int64_t* out;
  WsHeader* hdr;
  unsigned* rowkey;  // [rows]: largest published running maximum per row (order key; 0 none)
  TileSum* ts;     // [ntiles]
  float* slot_val;  // [ntiles, kSlotCap]
  int* slot_idx;
  float* pool_val;  // [pool_cap]
  int* pool_idx;
  unsigned pool_cap;
};

// One row's sampling parameters and what follows from them.
struct RowParams {
  float T, tp, mp;
  int k;
  bool greedy, has_p, has_m, has_k0, unfiltered, compact;
  float c2;     // log2(e) / T
  float tl;     // min-p bound below the maximum: max + tl
  float delta;  // compaction window below the running maximum
};

struct RawParams {
  float T, tp, mp;
  int k;
};
// Row `row`'s parameters: its slot's, rps rows to a slot.
__device__ __forceinline__ RawParams raw_params(const SampleArgs& a, int row) {
  RawParams p;
  const int s = row / a.rps;
  p.T = a.temp ? a.temp[s] : a.temp_s;
  p.k = a.topk ? a.topk[s] : a.topk_s;
  p.tp = a.topp ? a.topp[s] : a.topp_s;
  p.mp = a.minp ? a.minp[s] : a.minp_s;
  return p;
}
// Row `row`'s Philox key: its own seed, or the call's.
__device__ __forceinline__ uint2 philox_key(const SampleArgs& a, int row) {
  const uint64_t seed = a.seeds ? a.seeds[row] : a.seed;
  return make_uint2(uint32_t(seed), uint32_t(seed >> 32));
}
__device__ __forceinline__ RowParams row_params(const RawParams& p) {
  RowParams r;
  r.T = p.T;
  r.k = p.k;
  r.tp = p.tp;
  r.mp = p.mp;
  r.greedy = !(r.T > 0.f) || r.k == 1;
  r.has_p = !r.greedy && r.tp < 1.f;
  r.has_m = !r.greedy && r.mp > 0.f;
  r.has_k0 = !r.greedy && r.k > 0;
  r.unfiltered = !r.greedy && !r.has_p && !r.has_m && !r.has_k0;
  r.compact = !r.greedy && !r.unfiltered;
  r.c2 = r.greedy ? 0.f : kLog2e / r.T;
  r.tl = r.has_m ? r.T * logf(r.mp) : 0.f;
  float d = INFINITY;
  if (r.has_m) d = fminf(d, -r.tl);
  if (r.has_p) d = fminf(d, r.T * (2.f + 2.5f * logf(1.f / fmaxf(1.f - r.tp, 1e-6f))));
  if (r.has_k0) d = fminf(d, kWindowK);
  r.delta = d > 0.f ? d : 0.f;
  return r;
}

// Gumbel score of candidate token v of row with z = x / T; w4/wgrp cache v's
// Philox block.
__device__ __forceinline__ float gumbel_score(float z, int v, int row, uint64_t offset,
                                             uint2 key, uint4& w4, int& wgrp) {
  const int grp = v >> 2;
  if (grp != wgrp) {
    w4 = philox4x32_10(
        make_uint4(uint32_t(grp), uint32_t(row), uint32_t(offset), uint32_t(offset >> 32)), key);
    wgrp = grp;
  }
  const uint32_t word = (v & 3) == 0 ? w4.x : (v & 3) == 1 ? w4.y : (v & 3) == 2 ? w4.z : w4.w;
  return z + gumbel_from_word(word);
}

// The Gumbel score of candidate v if it may reach `best`, else -inf, without the
// two logarithms for most tokens that cannot: with u the token's uniform,
// g = -log(w) and w = -log(u) >= 1 - u, so 1 - u > e^(z - best) (taken with a
// margin above the approximate exponential) proves z + g < best.  1 - u is exact
// in float.  Used only where best is a score already seen, so a skipped token
// can never be the draw.
__device__ __forceinline__ float gumbel_score_vs(float z, int v, int row, uint64_t offset,
                                                uint2 key, uint4& w4, int& wgrp, float best) {
  const int grp = v >> 2;
  if (grp != wgrp) {
    w4 = philox4x32_10(
        make_uint4(uint32_t(grp), uint32_t(row), uint32_t(offset), uint32_t(offset >> 32)), key);
    wgrp = grp;
  }
  const uint32_t word = (v & 3) == 0 ? w4.x : (v & 3) == 1 ? w4.y : (v & 3) == 2 ? w4.z : w4.w;
  if (best > -INFINITY) {
    const float one_minus_u = (float(8388608u - (word >> 9)) - 0.5f) * 1.1920928955078125e-07f;
    const float bound = ex2((z - best) * kLog2e) * 1.0001f;
    if (one_minus_u > bound) return -INFINITY;
  }
  return z + gumbel_from_word(word);
}

// x * (1 / T) is within 3 * 2^-24 relative of x / T; a bound widened by 2^-20 of
// |z| therefore holds for either.
constexpr float kZRel = 9.5367431640625e-07f;  // 2^-20

// gumbel_score_vs for logit x, with z = x / T formed only for a token that the
// skip test lets through: the test takes x * invT and a bound widened by kZRel,
// so a skipped token still provably cannot reach `best`, and the score of a
// token that is not skipped is the one gumbel_score_vs gives.
__device__ __forceinline__ float gumbel_score_vx(float x, float T, float invT, int v, int row,
                                                uint64_t offset, uint2 key, uint4& w4, int& wgrp,
                                                float best) {
  const int grp = v >> 2;
  if (grp != wgrp) {
    w4 = philox4x32_10(
        make_uint4(uint32_t(grp), uint32_t(row), uint32_t(offset), uint32_t(offset >> 32)), key);
    wgrp = grp;
  }
  const uint32_t word = (v & 3) == 0 ? w4.x : (v & 3) == 1 ? w4.y : (v & 3) == 2 ? w4.z : w4.w;
  if (best > -INFINITY) {
    const float za = x * invT;
    const float one_minus_u = (float(8388608u - (word >> 9)) - 0.5f) * 1.1920928955078125e-07f;
    const float bound = ex2((za - best + fabsf(za) * kZRel) * kLog2e) * 1.0001f;
    if (one_minus_u > bound) return -INFINITY;
  }
  return __fdiv_rn(x, T) + gumbel_from_word(word);
}

// Programmatic dependent launch: wait for the grid this one depends on, and let
// the next grid in the stream begin its launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Radix histograms, double-buffered by pass parity.  A bin's mass (a sum of
// 2^-40 fixed-point masses, each at most 2^40) is kept exactly in three 32-bit
// limbs of 14, 14 and 13 bits per addend, since 64-bit shared-memory atomics are
// far slower than 32-bit ones; a limb cannot overflow while a bin takes at most
// kLimbRows addends per pass.  Rows with more candidates use 64-bit atomics.
constexpr unsigned kLimbRows = 1u << 18;
struct Hist {
  union {
    unsigned long long mass[2][256];
    unsigned limb[2][256][3];
  };
  unsigned cnt[2][256];
};
__device__ __forceinline__ void limb_add(unsigned* l, unsigned long long m) {
  atomicAdd(l, unsigned(m & 0x3FFFu));
  atomicAdd(l + 1, unsigned((m >> 14) & 0x3FFFu));
  atomicAdd(l + 2, unsigned(m >> 28));
}
__device__ __forceinline__ unsigned long long limb_sum(const unsigned* l) {
  return static_cast<unsigned long long>(l[0]) + (static_cast<unsigned long long>(l[1]) << 14) +
         (static_cast<unsigned long long>(l[2]) << 28);
}

__device__ __forceinline__ void arg_combine(float& s, int& v, float s2, int v2) {
  if (s2 > s || (s2 == s && v2 < v)) {
    s = s2;
    v = v2;
  }
}

// Merge two partial summaries (max, lowest index of the max and -- when
// with_sum -- the sum of exp2((x - max) c2)).  Symmetric in its two arguments, so
// a butterfly leaves the same value in every lane and any fixed merge order is
// deterministic.
__device__ __forceinline__ void row_combine(float& m, int& v, float& s, float m2, int v2, float s2,
                                            float c2, bool with_sum) {
  if (with_sum) {
    const float M = fmaxf(m, m2);
    const float a = m > -INFINITY ? s * ex2((m - M) * c2) : 0.f;
    const float b = m2 > -INFINITY ? s2 * ex2((m2 - M) * c2) : 0.f;
    s = a + b;
  }
  arg_combine(m, v, m2, v2);
}

// ------------------------------------------------------ TMA and mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* m, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(m)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Arrive once and add `bytes` to the phase's expected transaction count.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* m, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(m)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity to complete: a few
// non-blocking tests first (a phase that completes soon is seen without a
// suspend and wake-up), then try_wait, which suspends the thread for a
// hardware-chosen time slice; after kMaxWaitTries failures (far beyond any
// copy's latency) it gives up and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity) {
  for (int i = 0; i < kTestWaits; ++i)
    if (mbar_test_wait(m, parity)) return true;
  for (uint32_t i = 0; i < kMaxWaitTries; ++i)
    if (mbar_try_wait(m, parity)) return true;
  return false;
}
// One-dimensional bulk copy global -> shared completing on mbarrier m; both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* m) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(m))
      : "memory");
}

// -------------------------------------------------------------- row span

// A contiguous span of one row (a tile, or the whole row): local element i is
// token start + i, at byte mis + i * EB of a 16-byte aligned window starting at
// g0.  The window is streamed in pieces of kPieceBytes.  Whole 16-byte vectors
// [qf0, qf1) of the window arrive by bulk copy; the ragged first and last
// vectors are read from global memory when used.  Each piece's bitmask words
// arrive with it: words [m_lo, m_hi) (relative to the span) sit at byte
// 4 (w - m_lo) of the piece's mask slot; other words are read from global
// memory.
template <int DT>
struct Span {
  using E = Elt<DT>;
  static constexpr int EPV = E::kPerVec;
  static constexpr int EB = E::kBytes;
  static constexpr uint32_t ALL = (1u << EPV) - 1u;
  const char* g0;
  const uint32_t* gmask;  // the span's bitmask words (masked rows)
  int start, n_local, mis, win, nvec, nwords, qf0, qf1, npieces;
  bool masked;

  // tokens [s, s + n) of row (s a multiple of 32)
  __device__ __forceinline__ void init(const SampleArgs& a, int row, int s, int n, bool m) {
    start = s;
    n_local = max(0, n);
    const char* gsrc = a.logits + int64_t(row) * a.stride_bytes + int64_t(start) * EB;
    mis = int(reinterpret_cast<uintptr_t>(gsrc) & 15);
    g0 = gsrc - mis;
    win = mis + n_local * EB;
    nvec = n_local ? (win + 15) >> 4 : 0;
    qf0 = (mis + 15) >> 4;
    qf1 = win >> 4;
    nwords = (n_local + 31) >> 5;
    npieces = n_local ? (win + kPieceBytes - 1) / kPieceBytes : 0;
    masked = m;
    gmask = m ? a.bitmask + int64_t(row) * a.bm_stride + (start >> 5) : nullptr;
  }
  // tile `part` of row
  __device__ __forceinline__ void init_tile(const SampleArgs& a, int row, int part, bool m) {
    const int s = part * a.chunk;
    init(a, row, s, min(a.chunk, a.V - s), m);
  }
  // vectors [q0, q1) of piece j
  __device__ __forceinline__ void piece_vecs(int j, int& q0, int& q1) const {
    q0 = j * (kPieceBytes / 16);
    q1 = min(q0 + kPieceBytes / 16, nvec);
  }
  // bitmask words [w0, w1) the vectors of piece j touch
  __device__ __forceinline__ void piece_words(int j, int& w0, int& w1) const {
    int q0, q1;
    piece_vecs(j, q0, q1);
    const int i0 = max((16 * q0 - mis) / EB, 0);
    const int i1 = min((16 * q1 - mis) / EB, n_local);  // exclusive
    w0 = i0 >> 5;
    w1 = i1 > i0 ? ((i1 - 1) >> 5) + 1 : w0;
  }
  // the 16-byte aligned interior [m_lo, m_hi) of words [w0, w1)
  __device__ __forceinline__ void mask_interior(int w0, int w1, int& m_lo, int& m_hi) const {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(gmask + w0);
    const int lead = int(((16 - (a0 & 15)) & 15) >> 2);
    m_lo = min(w0 + lead, w1);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(gmask + w1) & ~uintptr_t(15);
    m_hi = max(m_lo, int((a1 - reinterpret_cast<uintptr_t>(gmask)) >> 2));
  }
  __device__ __forceinline__ uint4 gvec(int q) const {  // from global memory
    if (q >= qf0 && q < qf1) return __ldg(reinterpret_cast<const uint4*>(g0 + 16 * q));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int off = 16 * q + e * EB;
      if (off >= mis && off < win) {
        const uint32_t b = E::bits1(g0 + off);
        if (EB == 4)
          w[e] = b;
        else
          w[e >> 1] |= b << (16 * (e & 1));
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  // candidate bits of vector q (element e a token of this span kept by the
  // mask), its mask words taken from `mw` (words [m_lo, m_hi)) or global memory
  __device__ __forceinline__ uint32_t bits(int q, int& i0, const uint32_t* mw, int m_lo,
                                           int m_hi) const {
    i0 = (16 * q - mis) / EB;
    uint32_t valid = ALL;
    if (i0 < 0 || i0 + EPV > n_local) {
      const int lo = i0 < 0 ? -i0 : 0;
      const int hi = min(EPV, n_local - i0);
      valid = hi > lo ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
    }
    if (!masked || !valid) return valid;
    const int w = i0 >> 5;  // floor division: -1 for a negative i0
    const int sh = i0 & 31;
    auto word = [&](int x) -> uint32_t {
      return (x >= m_lo && x < m_hi) ? mw[x - m_lo] : __ldg(gmask + x);
    };
    const uint32_t w0 = w >= 0 ? word(w) : 0u;
    const uint32_t w1 = (sh + EPV > 32 && w + 1 < nwords) ? word(w + 1) : 0u;
    return valid & uint32_t(((uint64_t(w1) << 32) | w0) >> sh);
  }
};

// Rows listed in the call's indices (every row when there is no list) are
// masked; block-uniform, every thread of the block calls it.
__device__ __forceinline__ bool row_masked(const SampleArgs& a, int row) {
  if (!a.bitmask) return false;
  if (a.indices == nullptr) return true;
  int found = 0;
  for (int i = threadIdx.x; i < a.n_indices; i += blockDim.x) found |= (a.indices[i] == row);
  return __syncthreads_or(found) != 0 && row < a.bm_rows;
}

// ================================================================ stream kernel

// Bounded poll of a shared-memory hand-over counter: true once *p == target,
// false after `limit` polls of 64 ns sleeps.
constexpr uint32_t kFreshPolls = kMaxWaitTries * 64u;
__device__ __forceinline__ bool poll_fresh(const int* p, int target, uint32_t limit) {
  for (uint32_t t = 0; *(const volatile int*)p != target; ++t) {
    if (t >= limit) return false;
    __nanosleep(64);
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* m) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(m)) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) sample_stream_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  using Sp = Span<DT>;
  constexpr int EPV = E::kPerVec;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* const ring = smem;
  unsigned char* const mring = smem + kRing * kPieceBytes;
  // compaction buffers, one per tile parity: the value and the token's offset
  // into the tile
  using Cp = Compact<DT>;
  using CVal = typename Cp::Val;
  constexpr int kCapT = Cp::kCapT;
  CVal* const bval0 = reinterpret_cast<CVal*>(mring + kRing * kMaskSlot);
  uint16_t* const bidx0 = reinterpret_cast<uint16_t*>(bval0 + 2 * kCapT);

  // Per-tile state, double-buffered by tile parity: the warps of a CTA finish a
  // tile independently; the last one to finish it merges the warps' partial
  // summaries, writes the tile out and readies the parity for tile it + 2.
  __shared__ float red_f[2][kConsumerWarps], red_s[2][kConsumerWarps], red_b[2][kConsumerWarps];
  __shared__ int red_i[2][kConsumerWarps], red_n[2][kConsumerWarps], red_bv[2][kConsumerWarps];
  __shared__ int s_count[2], s_done[2], s_fresh[2], s_err;
  __shared__ unsigned s_runkey[2];
  __shared__ __align__(8) uint64_t full[kRing];
  __shared__ __align__(8) uint64_t empty[kRing];
  __shared__ uint4 keep_tab[256];  // 16-bit types: per-word keep masks of 8 element bits
  __shared__ int4 pmeta[kRing];    // per slot: vectors [x, y), staged mask words [z, w)
  __shared__ int pflag[kRing];     // per slot: bit 0 whole vectors only, bit 1 row masked
  __shared__ uint2 pkey[kRing];    // per slot: the Philox key of the piece's row

  if (tid == 0) {
    s_err = 0;
    for (int p = 0; p < 2; ++p) {
      s_count[p] = 0;
      s_done[p] = 0;
      s_runkey[p] = 0u;
      s_fresh[p] = p;  // parity p is ready for tile iteration p
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&full[r], 1);
      mbar_init(&empty[r], kConsumerWarps);
    }
    mbar_init_fence();
  }
  keep_tab[tid] = make_uint4(keep_mask16(tid, 0), keep_mask16(tid, 1), keep_mask16(tid, 2),
                             keep_mask16(tid, 3));
  // The finish kernel may begin its launch now; its blocks wait for this grid
  // to complete before they read anything.  This grid in turn waits for the
  // previous one in the stream before its first global read.
  launch_dependents();
  grid_dependency_wait();
  __syncthreads();

  // tiles per launch fit in 32 bits (at most kMaxTileSums)
  const unsigned G = gridDim.x, ntiles = unsigned(a.ntiles), tpr = unsigned(a.tpr);
  auto tile_of = [&](int it) { return blockIdx.x + unsigned(it) * G; };
  auto row_of = [&](unsigned t) { return a.row0 + int(t / tpr); };
  auto part_of = [&](unsigned t) { return int(t % tpr); };

  // ================================================================ producer
  // Warp kConsumerWarps copies the pieces of this CTA's tiles, in order, into
  // ring slot (n % kRing) of the n-th piece: it waits until the consumers have
  // released the slot, publishes the piece's geometry and starts its bulk
  // copies on the slot's mbarrier.
  if (warp == kConsumerWarps) {
    uint32_t issued = 0;
    for (int it = 0; tile_of(it) < ntiles; ++it) {
      const unsigned tile = tile_of(it);
      const int row = row_of(tile);
      bool masked = false;  // warp-uniform
      if (a.bitmask) {
        if (a.indices == nullptr) {
          masked = true;
        } else {
          int found = 0;
          for (int i = lane; i < a.n_indices; i += 32) found |= (a.indices[i] == row);
          masked = __any_sync(kFullWarp, found) && row < a.bm_rows;
        }
      }
      Sp g;
      g.init_tile(a, row, part_of(tile), masked);
      const uint2 rkey = philox_key(a, row);
      for (int j = 0; j < g.npieces; ++j, ++issued) {
        const int slot = int(issued % kRing);
        if (issued >= uint32_t(kRing) &&
            !mbar_wait(&empty[slot], ((issued / kRing) - 1u) & 1u) && lane == 0)
          s_err = 1;  // the consumers are gone: copy nothing more
        int q0, q1;
        g.piece_vecs(j, q0, q1);
        const int v0 = max(q0, g.qf0), v1 = min(q1, g.qf1);
        const uint32_t vbytes = v1 > v0 ? uint32_t(16 * (v1 - v0)) : 0u;
        uint32_t mbytes = 0;
        int base = 0, w1 = 0, m_lo = 0;
        if (g.masked) {
          // The slot holds the piece's words [w0, w1) from the 16-byte aligned
          // word base <= w0 on: the aligned interior by bulk copy, the (at most
          // three) words at each edge by plain loads of lanes 1-6.
          int w0, m_hi;
          g.piece_words(j, w0, w1);
          g.mask_interior(w0, w1, m_lo, m_hi);
          base = w0 - int((reinterpret_cast<uintptr_t>(g.gmask + w0) & 15) >> 2);
          mbytes = uint32_t(4 * (m_hi - m_lo));
          uint32_t* mslot = reinterpret_cast<uint32_t*>(mring + slot * kMaskSlot);
          const int x = lane >= 1 && lane <= 3 ? w0 + lane - 1
                        : lane >= 4 && lane <= 6 ? m_hi + lane - 4
                                                 : -1;
          if (x >= 0 && (lane <= 3 ? x < m_lo : x < w1)) mslot[x - base] = __ldg(g.gmask + x);
          __syncwarp();  // the edge words are stored before lane 0's arrive publishes them
        }
        if (lane != 0) continue;
        pmeta[slot] = make_int4(q0, q1, base, w1);  // published by the arrive below
        pflag[slot] = (q0 >= g.qf0 && q1 <= g.qf1 ? 1 : 0) | (g.masked ? 2 : 0);
        pkey[slot] = rkey;
        if (*(volatile int*)&s_err) {  // a copy went missing: start no more (rows report -2)
          mbar_expect_tx(&full[slot], 0);
          continue;
        }
        mbar_expect_tx(&full[slot], vbytes + mbytes);
        if (vbytes)
          bulk_load(ring + slot * kPieceBytes + 16 * (v0 - q0), g.g0 + 16 * v0, vbytes,
                    &full[slot]);
        if (mbytes)
          bulk_load(mring + slot * kMaskSlot + 4 * (m_lo - base), g.gmask + m_lo, mbytes,
                    &full[slot]);
      }
    }
    return;
  }

  // =============================================================== consumers
  uint32_t consumed = 0, lost = 0;
  RawParams nxt{};  // the next tile's row parameters, loaded a tile ahead
  if (tile_of(0) < ntiles) nxt = raw_params(a, row_of(tile_of(0)));

  for (int it = 0; tile_of(it) < ntiles; ++it) {
    const unsigned tile = tile_of(it);
    const int row = row_of(tile);
    const int lrow = row - a.row0;
    const int par = it & 1;
    CVal* const bval = bval0 + par * kCapT;
    uint16_t* const bidx = bidx0 + par * kCapT;

    Sp pt;
    pt.init_tile(a, row, part_of(tile), false);  // masked: from the first piece
    const RowParams rp = row_params(nxt);
    if (tile_of(it + 1) < ntiles) nxt = raw_params(a, row_of(tile_of(it + 1)));
    const float T = rp.T, c2 = rp.c2, delta = rp.delta;

    // this parity's state is ready once the last warp of tile it - 2 has reset
    // it (bounded wait; the warps of a CTA are at most a few pieces apart).  A
    // wait that gives up marks the CTA's tiles from here on as failed (their
    // rows report -2), then waits once more, also bounded, so that the state is
    // still left alone until it is handed over.
    if (lane == 0) {
      bool ok = poll_fresh(&s_fresh[par], it, kFreshPolls);
#ifdef LP_TEST_FRESH_TIMEOUT
      // test builds only: one wait of CTA 0 polls for a hand-over that never
      // comes, LP_TEST_FRESH_TIMEOUT times, and so runs out
      if (ok && blockIdx.x == 0 && it == 1)
        ok = poll_fresh(&s_fresh[par], it + (1 << 30), LP_TEST_FRESH_TIMEOUT);
#endif
      if (!ok) {
        s_err = 1;
        (void)poll_fresh(&s_fresh[par], it, kFreshPolls);
      }
      __threadfence_block();
    }
    __syncwarp();

    // the largest running maximum the row's other tiles have published, read one
    // piece ahead of its use (thread 0); the largest key this lane has published
    unsigned hint = 0u, wpub = 0u;

    // ------------------------------------------------------ stream the tile
    float m = -INFINITY, sm = 0.f;  // running max and softmax sum relative to it
    int targ = INT_MAX, cnt = 0;    // lowest index of the running max; candidate bits seen
    float best = -INFINITY;         // unfiltered rows: running best score
    int bestv = INT_MAX;
    uint4 w4 = make_uint4(0, 0, 0, 0);
    int wgrp = -1;
    bool stream_ok = true;
    // The piece loop, compiled once per row mode so that each mode's loop holds
    // only its own work.
    auto stream = [&](auto mode_tag) {
      constexpr int kMode = decltype(mode_tag)::value;
      constexpr bool has_p = kMode == kModeTopP;
      constexpr bool unfiltered = kMode == kModeUnfiltered;
      constexpr bool compact = kMode == kModeTopP || kMode == kModeFilter;
      for (int j = 0; j < pt.npieces; ++j) {
        const int slot = int(consumed % kRing);
        const uint32_t parity = (consumed / kRing) & 1u;
        ++consumed;
        if (!mbar_wait(&full[slot], parity)) {
          stream_ok = false;
          s_err = 1;
          lost |= (1u << slot) | (parity << (slot + 8));
        }
        const int4 pm = pmeta[slot];
        const int pf = pflag[slot];
        const bool whole = (pf & 1) != 0;
        if (j == 0 && (pf & 2)) {
          pt.masked = true;
          pt.gmask = a.bitmask + int64_t(row) * a.bm_stride + (pt.start >> 5);
        }
        const unsigned char* data = ring + slot * kPieceBytes;
        const uint32_t* mw = reinterpret_cast<const uint32_t*>(mring + slot * kMaskSlot);
        // vector q of this piece and its candidate bits
        const bool plain = whole && !pt.masked;  // every vector staged, every token a candidate
        // whole vectors of an aligned span: a vector's bits sit in one staged word
        const bool aligned = whole && pt.masked && pt.mis == 0;
        // vector q of this piece (its staged copy already in raw) and its candidate bits
        auto load = [&](int q, uint4& raw, uint32_t& cb) {
          if (plain) {
            cb = Sp::ALL;
            return;
          }
          if (aligned) {
            const int i0 = q * EPV;
            cb = (mw[(i0 >> 5) - pm.z] >> (i0 & 31)) & Sp::ALL;
            return;
          }
          if (!whole && !(q >= pt.qf0 && q < pt.qf1)) raw = pt.gvec(q);  // a ragged edge
          int i0;
          cb = pt.bits(q, i0, mw, pm.z, pm.w);
        };
        // the vector with every non-candidate element replaced by -inf
        auto masked_vec = [&](const uint4& raw, uint32_t cb) -> uint4 {
          if (cb == Sp::ALL) return raw;
          if (Sp::EB == 4) {
            constexpr uint32_t kNegInf = 0xff800000u;
            return make_uint4((cb & 1u) ? raw.x : kNegInf, (cb & 2u) ? raw.y : kNegInf,
                              (cb & 4u) ? raw.z : kNegInf, (cb & 8u) ? raw.w : kNegInf);
          }
          const uint32_t ninf2 = DT == LP_BF16 ? 0xff80ff80u : 0xfc00fc00u;
          const uint4 t = keep_tab[cb];
          return make_uint4((raw.x & t.x) | (ninf2 & ~t.x), (raw.y & t.y) | (ninf2 & ~t.y),
                            (raw.z & t.z) | (ninf2 & ~t.z), (raw.w & t.w) | (ninf2 & ~t.w));
        };
        // every vector of the thread first (independent loads and maxima), then the
        // running maximum once, then the softmax terms
        uint4 mv[kPerPiece];
        uint32_t cbs[kPerPiece];
        float vms[kPerPiece];
        // the staged vectors sit at fixed offsets of the slot: load them before the
        // piece's geometry is known
        uint4 stg[kPerPiece];
#pragma unroll
        for (int r = 0; r < kPerPiece; ++r)
          stg[r] = *reinterpret_cast<const uint4*>(data + 16 * (r * kConsumers + tid));
#pragma unroll
        for (int r = 0; r < kPerPiece; ++r) {
          const int q = pm.x + r * kConsumers + tid;
          uint4 raw = stg[r];
          uint32_t cb = 0;
          if (q < pm.y) load(q, raw, cb);
          cbs[r] = cb;
          mv[r] = masked_vec(raw, cb);
          vms[r] = cb ? VecMax<DT>::run(mv[r], Sp::ALL) : -INFINITY;
          cnt += __popc(cb);
        }
        float pmx = vms[0];
        int rmx = 0;
#pragma unroll
        for (int r = 1; r < kPerPiece; ++r)
          if (vms[r] > pmx) {
            pmx = vms[r];
            rmx = r;
          }
        if (pmx > m) {  // a new running maximum: its lowest index in this piece
          if constexpr (has_p) sm *= ex2((m - pmx) * c2);  // 0 while m is still -inf
          m = pmx;
          uint4 best_v = mv[0];  // mv[rmx], without a run-time index
#pragma unroll
          for (int r = 1; r < kPerPiece; ++r)
            if (rmx == r) best_v = mv[r];
          const int q = pm.x + rmx * kConsumers + tid;
          const int i0 = (16 * q - pt.mis) / Sp::EB;
#pragma unroll
          for (int e = EPV - 1; e >= 0; --e)
            if (E::get(best_v, e) == pmx) targ = pt.start + i0 + e;
        }
        if constexpr (has_p) {  // -inf elements add 0 (m is finite once any candidate is seen)
          const float off = m * c2;
#pragma unroll
          for (int r = 0; r < kPerPiece; ++r) {
            if (!cbs[r] || !(m > -INFINITY)) continue;
#pragma unroll
            for (int e = 0; e < EPV; ++e) sm += ex2(fmaf(E::get(mv[r], e), c2, -off));
          }
        }
        if constexpr (unfiltered) {
          const uint2 key = pkey[slot];  // the row's Philox key, published with the piece
          // the element loop is not unrolled: each Gumbel score inlines a Philox
          // block, and one copy per vector keeps the kernel's code small
#pragma unroll
          for (int r = 0; r < kPerPiece; ++r) {
            if (!cbs[r]) continue;
            const int q = pm.x + r * kConsumers + tid;
            const int i0 = (16 * q - pt.mis) / Sp::EB;
#pragma unroll 1
            for (int e = 0; e < EPV; ++e) {
              const float x = E::get(mv[r], e);
              if (!(x > -INFINITY)) continue;
              const float z = __fdiv_rn(x, T);
              if (z + kGumbelMax < best) continue;  // cannot win
              const int v = pt.start + i0 + e;
              arg_combine(best, bestv,
                          gumbel_score_vs(z, v, row, a.offset, key, w4, wgrp, best), v);
            }
          }
        }
        if constexpr (compact) {  // append the piece's candidates within the window
          // this lane's running maximum as an order key (0: none yet), published
          // to the CTA when it rises
          const unsigned wk = m > -INFINITY ? fkey(m) : 0u;
          if (wk > wpub) {
            atomicMax(&s_runkey[par], wk);
            wpub = wk;
          }
          if (tid == 0) {  // exchange with the row's other tiles
            if (j > 0 && hint) atomicMax(&s_runkey[par], hint);
            const unsigned mine = *(volatile unsigned*)&s_runkey[par];
            if (mine) atomicMax(&a.rowkey[lrow], mine);
            hint = *(volatile unsigned*)&a.rowkey[lrow];
          }
          const unsigned rk = max(wk, *(volatile unsigned*)&s_runkey[par]);
          // a buffer that has overflowed is flagged at the tile's end whatever else
          // is appended: stop appending
          const float cut = *(volatile int*)&s_count[par] > kCapT ? INFINITY
                            : rk                                   ? __fsub_rd(key_float(rk), delta)
                                                                   : -INFINITY;
#pragma unroll
          for (int r = 0; r < kPerPiece; ++r) {
            // a lane without a vector has vms = -inf, which must not pass a cut of -inf;
            // few lanes are live once the cut has risen, so each takes its own
            // places with one shared-memory atomic (no warp-wide scan)
            const bool live = vms[r] > -INFINITY && vms[r] >= cut;
            if (!live) continue;
            const int q = pm.x + r * kConsumers + tid;
            uint32_t pass = 0;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const float x = E::get(mv[r], e);
              if (x >= cut && x > -INFINITY) pass |= 1u << e;
            }
            int pos = atomicAdd(&s_count[par], __popc(pass));
            const int i0 = (16 * q - pt.mis) / Sp::EB;
            while (pass) {
              const int e = __ffs(pass) - 1;
              pass &= pass - 1;
              if (pos < kCapT) {
                bval[pos] = Cp::pack(mv[r], e);
                bidx[pos] = uint16_t(i0 + e);
              }
              ++pos;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the slot
      }

      // ---------------------------------------------------- warp epilogue
      // the warp's maximum, its lowest index and the count by redux; the softmax
      // sum rescaled to the warp maximum and summed in a fixed tree
      float wm, ws = sm, wb = best;
      int wv, wbv = bestv;
      int wn = int(__reduce_add_sync(kFullWarp, unsigned(cnt)));
      {
        const unsigned mk = __reduce_max_sync(kFullWarp, m > -INFINITY ? fkey(m) : 0u);
        wm = mk ? key_float(mk) : -INFINITY;
        wv = int(__reduce_min_sync(kFullWarp, unsigned(mk && m == wm ? targ : INT_MAX)));
      }
      if constexpr (has_p) {
        ws = m > -INFINITY ? sm * ex2((m - wm) * c2) : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) ws += __shfl_xor_sync(kFullWarp, ws, o);
      }
      if constexpr (unfiltered) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
          const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
          arg_combine(wb, wbv, b2, bv2);
        }
      }
      int last = 0;
      if (lane == 0) {
        red_f[par][warp] = wm;
        red_s[par][warp] = ws;
        red_i[par][warp] = wv;
        red_n[par][warp] = wn;
        red_b[par][warp] = wb;
        red_bv[par][warp] = wbv;
        __threadfence_block();
        last = atomicAdd(&s_done[par], 1) == kConsumerWarps - 1;
      }
      if (!__shfl_sync(kFullWarp, last, 0)) return;
      // ------------------------------- the last warp writes the tile out
      __threadfence_block();  // the other warps' summaries and buffer entries
      wm = -INFINITY, ws = 0.f, wb = -INFINITY;
      wv = INT_MAX, wn = 0, wbv = INT_MAX;
      if (lane < kConsumerWarps) {
        wm = red_f[par][lane];
        ws = red_s[par][lane];
        wv = red_i[par][lane];
        wn = red_n[par][lane];
        wb = red_b[par][lane];
        wbv = red_bv[par][lane];
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFullWarp, wm, o);
        const float s2 = __shfl_xor_sync(kFullWarp, ws, o);
        const int v2 = __shfl_xor_sync(kFullWarp, wv, o);
        wn += __shfl_xor_sync(kFullWarp, wn, o);
        row_combine(wm, wv, ws, m2, v2, s2, c2, has_p);
        const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
        const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
        arg_combine(wb, wbv, b2, bv2);
      }
      // Drop the entries below the final cut (the tile's maximum, or a larger one
      // of the row, less the window): they were appended under a lower running
      // maximum.  The survivors keep their order in the buffer.
      unsigned n = 0u;
      if constexpr (compact) {
        const unsigned cnt_all = unsigned(*(volatile int*)&s_count[par]);
        if (cnt_all <= unsigned(kCapT)) {
          unsigned fk = wm > -INFINITY ? fkey(wm) : 0u;
          fk = max(fk, *(volatile unsigned*)&s_runkey[par]);
          const float fcut_t = fk ? __fsub_rd(key_float(fk), delta) : -INFINITY;
          for (unsigned b0 = 0; b0 < cnt_all; b0 += 32) {
            const unsigned i = b0 + lane;
            CVal x{};
            uint16_t v = 0;
            const bool keep =
                i < cnt_all && (x = bval[i], v = bidx[i], Cp::unpack(x) >= fcut_t);
            const unsigned bal = __ballot_sync(kFullWarp, keep);
            __syncwarp();  // every lane has read its entry before any is overwritten
            if (keep) {
              const unsigned pos = n + unsigned(__popc(bal & ((1u << lane) - 1u)));
              bval[pos] = x;
              bidx[pos] = v;
            }
            n += unsigned(__popc(bal));
          }
          __syncwarp();
        } else {
          n = cnt_all;  // overflowed: flagged below
        }
      }
      // the buffer goes to the tile's slot, or to the pool when longer
      unsigned nf = n, off = 0u;
      if (lane == 0) {
        if constexpr (compact) {
          if (n > unsigned(kCapT)) {
            nf = kTileOverflow;
          } else if (n > unsigned(kSlotCap)) {
            off = atomicAdd(&a.hdr->pool_used, n);
            if (off > a.pool_cap || n > a.pool_cap - off) nf = kTileOverflow;
          }
        }
        if (!stream_ok || *(volatile int*)&s_err) nf |= kTileError;
      }
      nf = __shfl_sync(kFullWarp, nf, 0);
      off = __shfl_sync(kFullWarp, off, 0);
      if (!(nf & (kTileOverflow | kTileError))) {
        const bool in_slot = nf <= unsigned(kSlotCap);
        float* dv = in_slot ? a.slot_val + size_t(tile) * kSlotCap : a.pool_val + off;
        int* di = in_slot ? a.slot_idx + size_t(tile) * kSlotCap : a.pool_idx + off;
        for (unsigned i = lane; i < nf; i += 32) {
          dv[i] = Cp::unpack(bval[i]);
          di[i] = pt.start + int(bidx[i]);
        }
      }
      __syncwarp();  // every lane is done with the buffer before it is handed on
      if (lane == 0) {
        TileSum& t = a.ts[tile];
        t.max = wm;
        t.arg = wv;
        t.sum = ws;
        t.ncand = wn;
        t.best = wb;
        t.best_v = wbv;
        t.off = off;
        t.nf = nf;
        if (compact && wm > -INFINITY) atomicMax(&a.rowkey[lrow], fkey(wm));
        // ready this parity for tile it + 2
        s_count[par] = 0;
        s_runkey[par] = 0u;
        s_done[par] = 0;
        __threadfence_block();
        *(volatile int*)&s_fresh[par] = it + 2;
      }
      __syncwarp();
    };
    switch (rp.greedy ? kModeGreedy
            : rp.has_p ? kModeTopP
            : rp.compact ? kModeFilter
                         : kModeUnfiltered) {
      case kModeGreedy: stream(std::integral_constant<int, kModeGreedy>{}); break;
      case kModeTopP: stream(std::integral_constant<int, kModeTopP>{}); break;
      case kModeFilter: stream(std::integral_constant<int, kModeFilter>{}); break;
      default: stream(std::integral_constant<int, kModeUnfiltered>{}); break;
    }
  }

  // Leave only once every stage is idle: a stage whose wait timed out gets one
  // more bounded wait.
  for (int sl = 0; sl < kRing; ++sl)
    if ((lost >> sl) & 1u) (void)mbar_wait(&full[sl], (lost >> (sl + 8)) & 1u);
}

// ================================================================ finish kernel

// What a filtered row's merged summary fixes before any selection: the top-k
// that still filters, the min-p cut fm, a certified lower bound fcut of the
// keep-threshold, the lowest logit lo_w down to which the tiles' buffers hold
// every candidate, and the top-p mass target P in 2^-40 units.
struct RowBounds {
  int k;
  bool has_k;
  float fm, fcut, lo_w;
  unsigned long long P;
};
__device__ __forceinline__ RowBounds row_bounds(const RowParams& rp, float lmax, float S,
                                                int ncand_ub) {
  RowBounds b;
  b.k = rp.k;
  if (b.k > 0 && b.k >= ncand_ub) b.k = 0;  // keeps every candidate
  b.has_k = b.k > 0;
  b.fm = rp.has_m ? fminf(__fadd_ru(lmax, rp.tl), lmax) : -INFINITY;
  b.fcut = b.fm;
  if (rp.has_p) {  // t_p >= (1 - top_p) / ncand, as a logit
    float D = logf(float(ncand_ub) / (fmaxf(1.f - rp.tp, 1e-30f) * S));
    D = fmaxf(D, 0.f) * 1.001f + 1e-3f;
    b.fcut = fmaxf(b.fcut, __fsub_rd(lmax, rp.T * D));
  }
  // the compaction window is the narrowest of the filters' windows (with min-p
  // alone it ends exactly at fm)
  b.lo_w = __fsub_ru(lmax, rp.delta);
  b.P = 0ull;
  if (rp.has_p) {
    const float t = fmaxf(rp.tp, 0.f) * S * 1099511627776.0f;
    b.P = t >= 1.8e19f ? ~0ull : static_cast<unsigned long long>(t);
  }
  return b;
}

// Softmax mass of logit x in 2^-40 units (x <= lmax), as every selection counts it.
__device__ __forceinline__ unsigned long long mass40(float x, float lmax, float c2) {
  return __float2ull_rn(ex2((x - lmax) * c2) * 1099511627776.0f);
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) sample_finish_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  using Sp = Span<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int kLow = int(E::kLowKeyBit);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  extern __shared__ __align__(16) unsigned char fsmem[];
  float* const bval = reinterpret_cast<float*>(fsmem);         // [kStage]
  int* const bidx = reinterpret_cast<int*>(bval + kStage);     // [kStage]
  unsigned* const tstart = reinterpret_cast<unsigned*>(bidx + kStage);  // [kMetaCap + 1]
  __shared__ Hist hist;  // by radix-pass parity
  __shared__ float red_f[kWarps], red_s[kWarps], red_b[kWarps];
  __shared__ int red_i[kWarps], red_n[kWarps], red_bv[kWarps];
  __shared__ unsigned red_fl[kWarps], red_c[kWarps];
  __shared__ unsigned scan_c[kWarps];
  __shared__ unsigned long long scan_m[kWarps];
  __shared__ int s_sel, s_i[4];
  __shared__ unsigned s_pub;  // the row's published key, as the stream kernel left it
  __shared__ float s_f[2];
  __shared__ unsigned s_above_c, s_total, s_nst;
  __shared__ unsigned long long s_above_m;

  grid_dependency_wait();  // the stream kernel's summaries and buffers are complete
  // the stream kernel is done with the pool: hand it back empty to the next one
  if (blockIdx.x == 0 && tid == 0) a.hdr->pool_used = 0u;

  const int lrow = blockIdx.x;
  const int row = a.row0 + lrow;
  if (tid == 0) {  // the row's key, then back to zero for the next call
    s_pub = a.rowkey[lrow];
    a.rowkey[lrow] = 0u;
  }
  const uint2 key = philox_key(a, row);
  const RowParams rp = row_params(raw_params(a, row));
  const float T = rp.T, c2 = rp.c2;
  const float invT = 1.f / T;  // for skip tests only (scores divide by T)
  const bool has_p = rp.has_p;
  const int64_t t0 = int64_t(lrow) * a.tpr;
  const TileSum* rts = a.ts + t0;
  const bool meta = a.tpr <= kMetaCap;  // tile starts of the staged buffer fit

  // ------------------------------------------- merge the tile summaries
  // Thread tid takes a contiguous run of tiles in order, then a fixed tree over
  // the threads: a deterministic merge.  Buffered entries per tile are counted
  // for the staging below.  A row of at most 32 tiles is merged by warp 0 alone,
  // one tile a lane, by the same tree (the other warps would hold only
  // identities, whose merge changes nothing).
  if (a.tpr <= 32) {
    if (warp == 0) {
      float wm = -INFINITY, ws = 0.f, wb = -INFINITY;
      int wv = INT_MAX, wn = 0, wbv = INT_MAX;
      unsigned flags = 0u, nbuf = 0u;
      if (lane < a.tpr) {
        const TileSum st = rts[lane];
        wn = st.ncand;
        row_combine(wm, wv, ws, st.max, st.arg, st.sum, c2, has_p);
        arg_combine(wb, wbv, st.best, st.best_v);
        flags = st.nf & (kTileOverflow | kTileError);
        nbuf = (st.nf & (kTileOverflow | kTileError)) ? 0u : st.nf;
      }
      unsigned incl = nbuf;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFullWarp, incl, o);
        if (lane >= o) incl += y;
      }
      if (meta && lane < a.tpr) tstart[lane] = incl - nbuf;  // the tile's start
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFullWarp, wm, o);
        const float s2 = __shfl_xor_sync(kFullWarp, ws, o);
        const int v2 = __shfl_xor_sync(kFullWarp, wv, o);
        wn += __shfl_xor_sync(kFullWarp, wn, o);
        row_combine(wm, wv, ws, m2, v2, s2, c2, has_p);
        const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
        const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
        arg_combine(wb, wbv, b2, bv2);
        flags |= __shfl_xor_sync(kFullWarp, flags, o);
      }
      const unsigned tot = __shfl_sync(kFullWarp, incl, 31);
      if (lane == 0) {
        s_f[0] = wm;
        s_f[1] = ws;
        s_i[0] = wv;
        s_i[1] = wn;
        s_i[2] = wbv;
        s_i[3] = int(flags >> 30);  // bit 0 overflow, bit 1 error
        s_total = tot;
        if (meta) tstart[a.tpr] = tot;
      }
    }
    __syncthreads();
  } else {
    const int per = (a.tpr + kThreads - 1) / kThreads;
    const int tb = min(tid * per, a.tpr), te = min(tb + per, a.tpr);
    float wm = -INFINITY, ws = 0.f, wb = -INFINITY;
    int wv = INT_MAX, wn = 0, wbv = INT_MAX;
    unsigned flags = 0u, nbuf = 0u;
    for (int t = tb; t < te; ++t) {
      const TileSum st = rts[t];
      wn += st.ncand;
      row_combine(wm, wv, ws, st.max, st.arg, st.sum, c2, has_p);
      arg_combine(wb, wbv, st.best, st.best_v);
      flags |= st.nf & (kTileOverflow | kTileError);
      const unsigned n = (st.nf & (kTileOverflow | kTileError)) ? 0u : st.nf;
      if (meta) tstart[t] = n;  // the count, turned into a start below
      nbuf += n;
    }
    // exclusive scan of nbuf over the threads (tile order)
    unsigned incl = nbuf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(kFullWarp, incl, o);
      if (lane >= o) incl += y;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(kFullWarp, wm, o);
      const float s2 = __shfl_xor_sync(kFullWarp, ws, o);
      const int v2 = __shfl_xor_sync(kFullWarp, wv, o);
      wn += __shfl_xor_sync(kFullWarp, wn, o);
      row_combine(wm, wv, ws, m2, v2, s2, c2, has_p);
      const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
      const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
      arg_combine(wb, wbv, b2, bv2);
      flags |= __shfl_xor_sync(kFullWarp, flags, o);
    }
    if (lane == 31) red_c[warp] = incl;
    if (lane == 0) {
      red_f[warp] = wm;
      red_s[warp] = ws;
      red_i[warp] = wv;
      red_n[warp] = wn;
      red_b[warp] = wb;
      red_bv[warp] = wbv;
      red_fl[warp] = flags;
    }
    __syncthreads();
    unsigned base = incl - nbuf;
    for (int w = 0; w < warp; ++w) base += red_c[w];
    if (meta) {  // counts -> starts, in place
      unsigned pos = base;
      for (int t = tb; t < te; ++t) {
        const unsigned n = tstart[t];
        tstart[t] = pos;
        pos += n;
      }
    }
    if (warp == 0) {
      wm = -INFINITY, ws = 0.f, wb = -INFINITY;
      wv = INT_MAX, wn = 0, wbv = INT_MAX;
      flags = 0u;
      unsigned tot = 0u;
      if (lane < kWarps) {
        wm = red_f[lane];
        ws = red_s[lane];
        wv = red_i[lane];
        wn = red_n[lane];
        wb = red_b[lane];
        wbv = red_bv[lane];
        flags = red_fl[lane];
        tot = red_c[lane];
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFullWarp, wm, o);
        const float s2 = __shfl_xor_sync(kFullWarp, ws, o);
        const int v2 = __shfl_xor_sync(kFullWarp, wv, o);
        wn += __shfl_xor_sync(kFullWarp, wn, o);
        row_combine(wm, wv, ws, m2, v2, s2, c2, has_p);
        const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
        const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
        arg_combine(wb, wbv, b2, bv2);
        flags |= __shfl_xor_sync(kFullWarp, flags, o);
        tot += __shfl_xor_sync(kFullWarp, tot, o);
      }
      if (lane == 0) {
        s_f[0] = wm;
        s_f[1] = ws;
        s_i[0] = wv;
        s_i[1] = wn;
        s_i[2] = wbv;
        s_i[3] = int(flags >> 30);  // bit 0 overflow, bit 1 error
        s_total = tot;
        if (meta) tstart[a.tpr] = tot;
      }
    }
    __syncthreads();
  }
  const float lmax = s_f[0];
  const float S = s_f[1];
  const int ncand_ub = s_i[1];  // candidates counted by their bits (-inf included)
  const bool row_err = (s_i[3] >> 1) != 0;
  // A published key above the row's maximum can only be stale (a workspace whose
  // front was not zero when the call began): the cuts it raised may have dropped
  // candidates, so the row is read again as if a buffer had overflowed.
  const bool any_overflow = (s_i[3] & 1) != 0 || s_pub > (lmax > -INFINITY ? fkey(lmax) : 0u);
  const unsigned total = s_total;

  if (row_err || lmax == -INFINITY || rp.greedy || rp.unfiltered) {
    if (tid == 0)
      a.out[row] = row_err ? -2
                   : lmax == -INFINITY ? -1
                   : rp.greedy ? s_i[0]
                               : (s_i[2] == INT_MAX ? -1 : s_i[2]);
    return;
  }

  // ------------------------------------------------------- filter bounds
  const RowBounds bd = row_bounds(rp, lmax, S, ncand_ub);
  const int k = bd.k;
  const bool has_k = bd.has_k;
  const float fm = bd.fm, fcut = bd.fcut;
  const float lo_w = bd.lo_w;  // the tiles' buffers hold every candidate in [lo_w, lmax]

  // ------------------------------- stage the tiles' buffers in shared memory
  // Entry i of the row (tile order) sits in tile t with tstart[t] <= i <
  // tstart[t + 1]: independent loads, one per entry.
  auto fetch = [&](unsigned i, float& x, int& v) {
    int lo = 0, hi = a.tpr - 1;  // the last tile whose start is <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tstart[mid] <= i)
        lo = mid;
      else
        hi = mid - 1;
    }
    const unsigned j = i - tstart[lo];
    if (tstart[lo + 1] - tstart[lo] <= unsigned(kSlotCap)) {
      x = a.slot_val[(t0 + lo) * kSlotCap + j];
      v = a.slot_idx[(t0 + lo) * kSlotCap + j];
    } else {
      const unsigned off = rts[lo].off;
      x = a.pool_val[off + j];
      v = a.pool_idx[off + j];
    }
  };
  const bool flat = meta && !any_overflow;  // entries addressable by their row position
  const float lo_b = fmaxf(lo_w, fcut);      // nothing below can be kept
  // Stage the entries at or above lo_b (the only ones any pass counts) in
  // shared memory; when they do not fit, every pass reads the workspace.
  unsigned nst = 0;
  bool staged = false;
  if (flat) {
    if (tid == 0) s_nst = 0u;
    __syncthreads();
    for (unsigned b0 = unsigned(warp) * 32u; b0 < total; b0 += kThreads) {
      const unsigned i = b0 + lane;
      float x = 0.f;
      int v = 0;
      bool keep = false;
      if (i < total) {
        fetch(i, x, v);
        keep = x >= lo_b;
      }
      const unsigned bal = __ballot_sync(kFullWarp, keep);
      unsigned base = 0u;
      if (lane == 0 && bal) base = atomicAdd(&s_nst, unsigned(__popc(bal)));
      base = __shfl_sync(kFullWarp, base, 0);
      if (keep) {
        const unsigned pos = base + unsigned(__popc(bal & ((1u << lane) - 1u)));
        if (pos < unsigned(kStage)) {
          bval[pos] = x;
          bidx[pos] = v;
        }
      }
    }
    __syncthreads();
    nst = s_nst;
    staged = nst <= unsigned(kStage);
  }

  // The row's buffered entries: f(x, token, valid), warp-uniform; the staged
  // ones from shared memory, else all of them from the workspace.
  auto buffered = [&](auto&& f) {
    if (staged) {
      for (unsigned b0 = unsigned(warp) * 32u; b0 < nst; b0 += kThreads) {
        const unsigned i = b0 + lane;
        const bool ok = i < nst;
        f(ok ? bval[i] : 0.f, ok ? bidx[i] : 0, ok);
      }
      return;
    }
    if (flat) {
      for (unsigned b0 = unsigned(warp) * 32u; b0 < total; b0 += kThreads) {
        const unsigned i = b0 + lane;
        const bool ok = i < total;
        float x = 0.f;
        int v = 0;
        if (ok) fetch(i, x, v);
        f(x, v, ok);
      }
      return;
    }
    for (int t = 0; t < a.tpr; ++t) {
      const unsigned n = rts[t].nf;
      if (n & (kTileOverflow | kTileError)) continue;
      const bool in_slot = n <= unsigned(kSlotCap);
      const float* sv = in_slot ? a.slot_val + (t0 + t) * kSlotCap : a.pool_val + rts[t].off;
      const int* si = in_slot ? a.slot_idx + (t0 + t) * kSlotCap : a.pool_idx + rts[t].off;
      for (unsigned b0 = unsigned(warp) * 32u; b0 < n; b0 += kThreads) {
        const unsigned i = b0 + lane;
        const bool ok = i < n;
        f(ok ? sv[i] : 0.f, ok ? si[i] : 0, ok);
      }
    }
  };
  // Re-reads the whole row from global memory: f(raw, cb, i0) per vector,
  // warp-uniform.  Each thread loads the bitmask words and logits of kReread
  // vectors (independent loads) before it works on any of them, so the loads of
  // a pass overlap instead of running one round trip after another.
  Sp rw;
  bool rw_ready = false;
  constexpr int kReread = 2;
  auto reread = [&](auto&& f) {
    if (!rw_ready) {
      rw.init(a, row, 0, a.V, row_masked(a, row));
      rw_ready = true;
    }
    for (int base = 0; base < rw.nvec; base += kThreads * kReread) {
      uint4 raw[kReread];
      uint32_t cb[kReread];
#pragma unroll
      for (int u = 0; u < kReread; ++u) {
        const int q = base + u * kThreads + tid;
        int i0 = 0;
        cb[u] = 0u;
        raw[u] = make_uint4(0, 0, 0, 0);
        if (q < rw.nvec) {
          cb[u] = rw.bits(q, i0, nullptr, 0, 0);
          raw[u] = rw.gvec(q);
        }
      }
#pragma unroll
      for (int u = 0; u < kReread; ++u) {
        const int q = base + u * kThreads + tid;
        f(raw[u], cb[u], (16 * q - rw.mis) / Sp::EB);
      }
    }
  };

  // Stages the elements of vector `raw` whose bits are set in `inb` (element e is
  // token tok0 + e) at consecutive places of the stage, taken for the whole warp
  // with one shared-memory atomic: a per-lane count, a scan over the lanes, and
  // stores at fixed element indices.  Warp-uniform.  The order of staged entries
  // is immaterial (the selections count, the draw breaks ties by token).
  auto stage_vec = [&](const uint4& raw, uint32_t inb, int tok0) {
    const int c = __popc(inb);
    if (!__any_sync(kFullWarp, c != 0)) return;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullWarp, incl, o);
      if (lane >= o) incl += y;
    }
    unsigned base = 0u;
    if (lane == 31) base = atomicAdd(&s_nst, unsigned(incl));
    unsigned pos = __shfl_sync(kFullWarp, base, 31) + unsigned(incl - c);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      if ((inb >> e) & 1u) {
        if (pos < unsigned(kStage)) {
          bval[pos] = E::get(raw, e);
          bidx[pos] = tok0 + e;
        }
        ++pos;
      }
    }
  };

  // ---------------------------------- radix select of the threshold
  const unsigned long long P = bd.P;  // fixed-point top-p mass target
  // a radix pass keeps its bins' masses in 32-bit limbs unless the row has more
  // candidates than a limb can sum
  const bool limbs = unsigned(ncand_ub) <= kLimbRows;
  // the selection targets (a sample's are scaled versions of the row's)
  int sel_k = has_k ? k : 0;
  unsigned long long sel_P = P;
  int npass = 0;  // histogram parity
  // Largest key x >= key(lo) with count(>= x) >= k (top-k) or mass(>= x) >= P
  // (top-p), counting candidates of the tiles' buffers or of a re-read of the
  // row.  False when none exists.
  // Over [lo, hi], with above_c0 / above_m0 already counted above hi.
  // Narrows a descent over the buffered entries.  One pass sums the count, the
  // exact fixed-point mass and the smallest and largest key of the entries in
  // [lo, hi] per bin of kThreads bins of equal width in value (bin 0 at the
  // top); the range shrinks to the entries of the first bin from the top at
  // which a target is reached, and the entries above them are counted.  Bins of
  // equal width spread the entries over many addresses, where the first digits
  // of the key (sign and exponent bits) would put most of them in a few bins and
  // serialize the atomics.  Bins are monotone in the value, so the entries above
  // the bin's largest key are exactly those of the bins before it.  False when
  // no target is reached in [lo, hi].
  __shared__ unsigned s_kmin[kThreads], s_kmax[kThreads];
  __shared__ float s_nlo, s_nhi;
  auto narrow = [&](float& lo, float& hi, unsigned& above_c, unsigned long long& above_m) -> bool {
    const float top = fminf(hi, lmax);
    if (!(top > lo)) return true;  // a single value: nothing to narrow
    const float bpl = float(kThreads) / (top - lo);
    const int hp = npass & 1;
    ++npass;
    hist.cnt[hp][tid] = 0u;
    if (limbs) {
      hist.limb[hp][tid][0] = 0u;
      hist.limb[hp][tid][1] = 0u;
      hist.limb[hp][tid][2] = 0u;
    } else {
      hist.mass[hp][tid] = 0ull;
    }
    s_kmin[tid] = 0xffffffffu;
    s_kmax[tid] = 0u;
    if (tid == 0) s_sel = INT_MAX;
    __syncthreads();
    const float lo0 = lo;
    buffered([&](float x, int, bool ok) {
      if (!(ok && x >= lo0 && x <= top)) return;
      const int b = min(max(int((top - x) * bpl), 0), kThreads - 1);
      if (has_p) {
        const unsigned long long mm = mass40(x, lmax, c2);
        if (limbs)
          limb_add(hist.limb[hp][b], mm);
        else
          atomicAdd(&hist.mass[hp][b], mm);
      }
      atomicAdd(&hist.cnt[hp][b], 1u);
      const uint32_t kx = fkey(x);
      atomicMin(&s_kmin[b], kx);
      atomicMax(&s_kmax[b], kx);
    });
    __syncthreads();
    const unsigned c = hist.cnt[hp][tid];
    const unsigned long long m = limbs ? limb_sum(hist.limb[hp][tid]) : hist.mass[hp][tid];
    unsigned ic = c;
    unsigned long long im = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned yc = __shfl_up_sync(kFullWarp, ic, o);
      const unsigned long long ym = __shfl_up_sync(kFullWarp, im, o);
      if (lane >= o) {
        ic += yc;
        im += ym;
      }
    }
    if (lane == 31) {
      scan_c[warp] = ic;
      scan_m[warp] = im;
    }
    __syncthreads();
    for (int w = 0; w < warp; ++w) {
      ic += scan_c[w];
      im += scan_m[w];
    }
    const unsigned cc = above_c + ic;
    const unsigned long long cm = above_m + im;
    if (c > 0u && ((sel_k > 0 && cc >= unsigned(sel_k)) || (has_p && cm >= sel_P)))
      atomicMin(&s_sel, tid);
    __syncthreads();
    const int b = s_sel;
    if (b == INT_MAX) return false;
    if (tid == b) {
      s_above_c = cc - c;
      s_above_m = cm - m;
      s_nlo = key_float(s_kmin[b]);
      s_nhi = key_float(s_kmax[b]);
    }
    __syncthreads();
    above_c = s_above_c;
    above_m = s_above_m;
    lo = s_nlo;
    hi = s_nhi;
    __syncthreads();  // every thread has its copy before the shared words are reused
    return true;
  };

  auto descend = [&](bool from_buffers, float lo, uint32_t& out_key, float hi = INFINITY,
                     unsigned above_c0 = 0u, unsigned long long above_m0 = 0ull) -> bool {
    if (from_buffers && !narrow(lo, hi, above_c0, above_m0)) return false;
    const uint32_t klo = fkey(lo), khi = fkey(fminf(hi, lmax));
    const uint32_t diff = klo ^ khi;
    int top = diff ? 32 - __clz(diff) : kLow + 1;  // one past the highest differing bit
    top = max(top, kLow + 1);
    int shift = max(top - 8, kLow);
    uint32_t prefix = top >= 32 ? 0u : khi & ~((1u << top) - 1u);
    unsigned above_c = above_c0;
    unsigned long long above_m = above_m0;
    for (;;) {
      const int hp = npass & 1;
      ++npass;
      hist.cnt[hp][tid] = 0u;
      if (limbs) {
        hist.limb[hp][tid][0] = 0u;
        hist.limb[hp][tid][1] = 0u;
        hist.limb[hp][tid][2] = 0u;
      } else {
        hist.mass[hp][tid] = 0ull;
      }
      if (tid == 0) s_sel = -1;
      __syncthreads();
      const uint32_t himask = top >= 32 ? 0u : ~((1u << top) - 1u);
      const uint32_t dmask = (1u << (top - shift)) - 1u;
      // element x (when part) into its bin: one 32-bit atomic for the count and,
      // for top-p rows, three for the mass limbs (or one 64-bit atomic)
      auto add = [&](float x, bool part) {
        if (!(part && x >= lo && x <= hi)) return;
        const uint32_t kx = fkey(x);
        if (((kx ^ prefix) & himask) != 0u) return;
        const int d = int((kx >> shift) & dmask);
        if (has_p) {
          const unsigned long long mm = mass40(x, lmax, c2);
          if (limbs)
            limb_add(hist.limb[hp][d], mm);
          else
            atomicAdd(&hist.mass[hp][d], mm);
        }
        atomicAdd(&hist.cnt[hp][d], 1u);
      };
      if (from_buffers) {
        buffered([&](float x, int, bool ok) { add(x, ok); });
      } else {
        reread([&](const uint4& raw, uint32_t cb, int) {
          if (!__any_sync(kFullWarp, cb != 0)) return;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float x = E::get(raw, e);
            add(x, ((cb >> e) & 1u) && x > -INFINITY);
          }
        });
      }
      __syncthreads();
      // bin tid, then a descending inclusive scan over the bins
      const unsigned c = hist.cnt[hp][tid];
      const unsigned long long mass = limbs ? limb_sum(hist.limb[hp][tid]) : hist.mass[hp][tid];
      unsigned sc = c;
      unsigned long long smass = mass;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned yc = __shfl_down_sync(kFullWarp, sc, o);
        const unsigned long long ym = __shfl_down_sync(kFullWarp, smass, o);
        if (lane + o < 32) {
          sc += yc;
          smass += ym;
        }
      }
      if (lane == 0) {
        scan_c[warp] = sc;
        scan_m[warp] = smass;
      }
      __syncthreads();
      for (int w = warp + 1; w < kWarps; ++w) {
        sc += scan_c[w];
        smass += scan_m[w];
      }
      const unsigned cc = above_c + sc;
      const unsigned long long cm = above_m + smass;
      const bool okb =
          cc > 0u && ((sel_k > 0 && cc >= unsigned(sel_k)) || (has_p && cm >= sel_P));
      if (okb) atomicMax(&s_sel, tid);
      __syncthreads();
      const int sel = s_sel;
      if (sel < 0) return false;
      if (tid == sel) {
        s_above_c = cc - c;
        s_above_m = cm - mass;
      }
      __syncthreads();
      above_c = s_above_c;
      above_m = s_above_m;
      prefix |= uint32_t(sel) << shift;
      if (shift == kLow) {
        out_key = prefix;
        return true;
      }
      top = shift;
      shift = max(top - 8, kLow);
    }
  };


  // ---------------------- a window around the threshold (top-p rows, re-read)
  // Two re-reads of the row stand in for a radix pass per key digit.  The first
  // sums the candidates' softmax mass and count in kWinBins equal bins of
  // (lmax - x) down to fcut (fp32 sums; bin 0 next to the maximum); the bin where
  // the cumulative mass (or count, for top-k) reaches its target bounds, with
  // one bin of margin each side, a window [lo2, hi2).  The second sums the exact
  // count and fixed-point mass above hi2, stages the window's candidates, and
  // draws Gumbel-max over the candidates above the window (all of them are kept:
  // the threshold lies in the window) into pre_best / pre_bestv.  The exact
  // descent over the staged window, started from those sums, gives the
  // threshold; the draw then adds the window's kept entries.  False when the
  // window misses the threshold or does not fit (the caller then descends the
  // whole row, and pre_best is not used).
  float pre_best = -INFINITY;
  int pre_bestv = INT_MAX;
  auto window_select = [&](uint32_t& out_key) -> bool {
    if (!has_p || !(fcut > -INFINITY) || !(lmax > fcut)) return false;
    const float bpl = float(kWinBins) / (lmax - fcut);      // bins per logit
    float* wmass = reinterpret_cast<float*>(fsmem);         // [kWinBins]
    unsigned* wcnt = reinterpret_cast<unsigned*>(wmass + kWinBins);
    for (int i = tid; i < kWinBins; i += kThreads) {
      wmass[i] = 0.f;
      wcnt[i] = 0u;
    }
    __syncthreads();
    reread([&](const uint4& raw, uint32_t cb, int) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = E::get(raw, e);
        if (!((cb >> e) & 1u) || !(x >= fcut)) continue;
        const int bn = min(max(int((lmax - x) * bpl), 0), kWinBins - 1);
        atomicAdd(&wmass[bn], ex2((x - lmax) * c2));
        atomicAdd(&wcnt[bn], 1u);
      }
    });
    __syncthreads();
    // thread tid sums bins [tid * kWinPer, (tid + 1) * kWinPer); then an
    // inclusive scan over the threads; the first bin whose cumulative sum
    // reaches a target is bt
    constexpr int kWinPer = kWinBins / kThreads;
    double cm = 0.0;  // the bins' sums carry fp32 rounding; the window's margin absorbs it
    unsigned cc = 0u;
    for (int i = 0; i < kWinPer; ++i) {
      cm += double(wmass[tid * kWinPer + i]);
      cc += wcnt[tid * kWinPer + i];
    }
    const double mine_m = cm;
    const unsigned mine_c = cc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double ym = __shfl_up_sync(kFullWarp, cm, o);
      const unsigned yc = __shfl_up_sync(kFullWarp, cc, o);
      if (lane >= o) {
        cm += ym;
        cc += yc;
      }
    }
    __shared__ double s_wm[kWarps];
    __shared__ unsigned s_wc[kWarps];
    if (lane == 31) {
      s_wm[warp] = cm;
      s_wc[warp] = cc;
    }
    if (tid == 0) s_sel = INT_MAX;
    __syncthreads();
    for (int w = 0; w < warp; ++w) {
      cm += s_wm[w];
      cc += s_wc[w];
    }
    const double target_m = double(fmaxf(rp.tp, 0.f)) * double(S);
    if (cm >= target_m || (has_k && cc >= unsigned(k))) {
      // this thread's range reaches a target: find the first bin in it that does
      double pm = cm - mine_m;
      unsigned pc = cc - mine_c;
      int first = kWinPer - 1;
      for (int i = 0; i < kWinPer; ++i) {
        pm += double(wmass[tid * kWinPer + i]);
        pc += wcnt[tid * kWinPer + i];
        if (pm >= target_m || (has_k && pc >= unsigned(k))) {
          first = i;
          break;
        }
      }
      atomicMin(&s_sel, tid * kWinPer + first);
    }
    __syncthreads();
    const int bt = s_sel;
    if (bt == INT_MAX) return false;
    // the window: bins [bt - 1, bt + 1], as logits
    const float hi2 = bt >= 2 ? __fadd_ru(lmax, -float(bt - 1) / bpl) : INFINITY;
    const float lo2 = fmaxf(__fadd_rd(lmax, -float(bt + 2) / bpl), fcut);
    // exact count and mass above the window; the window's candidates staged; the
    // draw over the candidates above the window (and at or above the min-p cut)
    const float dcut = fmaxf(hi2, fm);
    unsigned ca = 0u;
    unsigned long long ma = 0ull;
    uint4 w4 = make_uint4(0, 0, 0, 0);
    int wgrp = -1;
    if (tid == 0) s_nst = 0u;
    __syncthreads();
    reread([&](const uint4& raw, uint32_t cb, int i0) {
      uint32_t inb = 0u;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = E::get(raw, e);
        const bool cand = ((cb >> e) & 1u) && x > -INFINITY;
        if (cand && x >= hi2) {
          ++ca;
          ma += mass40(x, lmax, c2);
          if (x >= dcut) {
            const float za = x * invT;  // the tests' stand-in for x / T
            if (!(za + fabsf(za) * kZRel + kGumbelMax < pre_best)) {
              const int v = rw.start + i0 + e;
              const float sc =
                  gumbel_score_vx(x, T, invT, v, row, a.offset, key, w4, wgrp, pre_best);
              if (sc > -INFINITY) arg_combine(pre_best, pre_bestv, sc, v);
            }
          }
        }
        if (cand && x >= lo2 && x < hi2) inb |= 1u << e;
      }
      stage_vec(raw, inb, rw.start + i0);
    });
    // block sums of the exact counts above the window
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      ca += __shfl_xor_sync(kFullWarp, ca, o);
      ma += __shfl_xor_sync(kFullWarp, ma, o);
    }
    if (lane == 0) {
      scan_c[warp] = ca;
      scan_m[warp] = ma;
    }
    __syncthreads();
    ca = 0u;
    ma = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      ca += scan_c[w];
      ma += scan_m[w];
    }
    const unsigned nwin = s_nst;
    __syncthreads();
    if (nwin > unsigned(kStage) || (has_k && ca >= unsigned(k)) || ma >= P) {
      pre_best = -INFINITY;  // the threshold is not in the window: nothing decided
      pre_bestv = INT_MAX;
      return false;
    }
    staged = true;
    nst = nwin;
    if (descend(true, lo2, out_key, hi2, ca, ma)) return true;
    staged = false;
    pre_best = -INFINITY;
    pre_bestv = INT_MAX;
    return false;
  };

  // At most one staged entry per thread: the threshold by counting.  Thread i
  // sums the count and mass of the staged entries at or above its own logit;
  // the threshold is the largest staged logit at which a target is reached --
  // the radix descent's answer, since counts and masses change only at entries.
  // False when no entry reaches a target.
  auto select_few = [&](uint32_t& out_key) -> bool {
    const bool mine = unsigned(tid) < nst;
    const float xi = mine ? bval[tid] : 0.f;
    if (has_p) hist.mass[0][tid] = mine ? mass40(xi, lmax, c2) : 0ull;
    __syncthreads();
    unsigned cnt = 0u;
    unsigned long long ms = 0ull;
    if (mine) {
      for (unsigned j = 0; j < nst; ++j) {
        if (bval[j] >= xi) {
          ++cnt;
          if (has_p) ms += hist.mass[0][j];
        }
      }
    }
    const bool hit = mine && ((sel_k > 0 && cnt >= unsigned(sel_k)) || (has_p && ms >= sel_P));
    const unsigned kk = __reduce_max_sync(kFullWarp, hit ? fkey(xi) : 0u);
    if (lane == 0) scan_c[warp] = kk;
    __syncthreads();
    unsigned top = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) top = max(top, scan_c[w]);
    __syncthreads();  // scan_c and hist are free again
    out_key = top;
    return top != 0u;
  };

  // ---------------- a row read once more, narrowed by a sample (buffers missed)
  // A strided sample of the row's vectors (kStage elements, a fraction fr of the
  // row) stands in for the row.  Its own threshold for scaled targets is a likely
  // lower bound b of the row's: for top-k a quarter more than k fr candidates;
  // for top-p the sample's mass less half the row's tail budget (S - P) scaled
  // by fr, so that the row's mass below b is likely within its budget.  When the
  // sample says that the candidates at or above b would fit in shared memory, one
  // pass over the row counts them and their mass exactly and stages them.  When
  // they reach a target (so the row's threshold is at least b) and fit, the
  // threshold is selected among them, and the draw takes them with no further
  // pass.  False otherwise (nothing is decided from the sample alone).
  auto sample_select = [&](uint32_t& out_key) -> bool {
    if (!rw_ready) {
      rw.init(a, row, 0, a.V, row_masked(a, row));
      rw_ready = true;
    }
    constexpr int per = kStage / EPV;  // sampled vectors
    if (rw.nvec < 4 * per) return false;
    const int sv = rw.nvec / per;  // sample stride, in vectors
    const double fr = double(per) / double(rw.nvec);  // the sampled fraction of the row
    // 1. the sampled vectors' candidates at or above fcut, staged
    if (tid == 0) s_nst = 0u;
    __syncthreads();
    for (int base = 0; base < per; base += kThreads) {
      const int si = base + tid;
      uint4 raw = make_uint4(0, 0, 0, 0);
      uint32_t cb = 0;
      int i0 = 0;
      if (si < per) {
        const int q = si * sv;
        cb = rw.bits(q, i0, nullptr, 0, 0);
        if (cb) raw = rw.gvec(q);
      }
      uint32_t inb = 0u;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = E::get(raw, e);
        if (((cb >> e) & 1u) && x > -INFINITY && x >= fcut) inb |= 1u << e;
      }
      stage_vec(raw, inb, rw.start + i0);
    }
    __syncthreads();
    nst = min(s_nst, unsigned(kStage));
    __syncthreads();
    if (nst == 0u) return false;
    staged = true;
    // 2. the sample's threshold for the scaled targets
    unsigned long long mt = 0ull;  // the sample's mass
    if (has_p) {
      for (unsigned i = unsigned(tid); i < nst; i += kThreads) mt += mass40(bval[i], lmax, c2);
#pragma unroll
      for (int o = 16; o; o >>= 1) mt += __shfl_xor_sync(kFullWarp, mt, o);
      if (lane == 0) scan_m[warp] = mt;
      __syncthreads();
      mt = 0ull;
      for (int w = 0; w < kWarps; ++w) mt += scan_m[w];
      __syncthreads();
    }
    const double budget = 0.5 * fr * (double(S) * 1099511627776.0 - double(P));
    sel_k = has_k ? int(fmin(ceil(1.25 * double(k) * fr) + 8.0, 2.0e9)) : 0;
    sel_P = has_p && double(mt) > budget ? static_cast<unsigned long long>(double(mt) - budget)
                                         : 0ull;
    uint32_t kb = 0;
    const bool got = (!has_p || sel_P > 0ull) &&
                     (nst <= unsigned(kThreads) ? select_few(kb) : descend(true, fcut, kb));
    sel_k = has_k ? k : 0;
    sel_P = P;
    if (!got) {
      staged = false;
      return false;
    }
    const float bnd = fmaxf(key_float(kb), fcut);
    // the sample's count at or above bnd, scaled: more than fits -> no pass
    unsigned cs = 0u;
    for (unsigned i = unsigned(tid); i < nst; i += kThreads) cs += bval[i] >= bnd ? 1u : 0u;
    cs = __reduce_add_sync(kFullWarp, cs);
    if (lane == 0) scan_c[warp] = cs;
    __syncthreads();
    cs = 0u;
    for (int w = 0; w < kWarps; ++w) cs += scan_c[w];
    __syncthreads();
    staged = false;
    if (double(cs) > 0.75 * double(kStage) * fr) return false;
    // 3. one pass: exact count and mass at or above bnd, those candidates staged
    unsigned ca = 0u;
    unsigned long long ma = 0ull;
    if (tid == 0) s_nst = 0u;
    __syncthreads();
    reread([&](const uint4& raw, uint32_t cb, int i0) {
      uint32_t inb = 0u;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = E::get(raw, e);
        if (((cb >> e) & 1u) && x > -INFINITY && x >= bnd) {
          inb |= 1u << e;
          ++ca;
          if (has_p) ma += mass40(x, lmax, c2);
        }
      }
      stage_vec(raw, inb, rw.start + i0);
    });
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      ca += __shfl_xor_sync(kFullWarp, ca, o);
      ma += __shfl_xor_sync(kFullWarp, ma, o);
    }
    if (lane == 0) {
      scan_c[warp] = ca;
      scan_m[warp] = ma;
    }
    __syncthreads();
    ca = 0u;
    ma = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      ca += scan_c[w];
      ma += scan_m[w];
    }
    const unsigned n = s_nst;
    __syncthreads();
    if (n > unsigned(kStage)) return false;                       // too many to stage
    if (!((has_k && ca >= unsigned(k)) || (has_p && ma >= P))) return false;  // b too high
    // 4. the threshold among them
    nst = n;
    staged = true;
    if (nst <= unsigned(kThreads) ? select_few(out_key) : descend(true, bnd, out_key)) return true;
    staged = false;
    return false;
  };

  float thr = fm;
  bool from_buffers = !any_overflow;
  if (has_k || has_p) {
    uint32_t kx = 0;
    bool found = false;
    if (from_buffers) {
      found = staged && nst <= unsigned(kThreads) ? select_few(kx) : descend(true, lo_b, kx);
      if (!found && !(fm >= lo_b)) from_buffers = false;
    }
    if (!from_buffers) {
      if (sample_select(kx) || window_select(kx)) {
        // every kept candidate is staged (the window's, with the ones above it
        // drawn already into pre_best): the draw takes them
        found = true;
        from_buffers = true;
      } else {
        found = descend(false, fcut, kx);
      }
    }
    if (found) thr = fmaxf(key_float(kx), fm);
  } else if (from_buffers && !(fm >= lo_w)) {
    from_buffers = false;
  }

  // ----------------------------------------------------------------- draw
  float best = pre_best;  // the window search's draw above its window, if any
  int bestv = pre_bestv;
  if (from_buffers) {
    buffered([&](float x, int v, bool ok) {
      if (!ok || !(x >= thr)) return;
      uint4 w;
      int g = -1;
      arg_combine(best, bestv, gumbel_score(__fdiv_rn(x, T), v, row, a.offset, key, w, g), v);
    });
  } else {
    uint4 w4 = make_uint4(0, 0, 0, 0);
    int wgrp = -1;
    reread([&](const uint4& raw, uint32_t cb, int i0) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = E::get(raw, e);
        if (!((cb >> e) & 1u) || !(x >= thr) || !(x > -INFINITY)) continue;
        const float za = x * invT;  // the tests' stand-in for x / T
        if (za + fabsf(za) * kZRel + kGumbelMax < best) continue;
        const int v = rw.start + i0 + e;
        arg_combine(best, bestv,
                    gumbel_score_vx(x, T, invT, v, row, a.offset, key, w4, wgrp, best), v);
      }
    });
  }
  {
    float wb = best;
    int wbv = bestv;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
      const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
      arg_combine(wb, wbv, b2, bv2);
    }
    if (lane == 0) {
      red_b[warp] = wb;
      red_bv[warp] = wbv;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float wb = -INFINITY;
    int wbv = INT_MAX;
    for (int w = 0; w < kWarps; ++w) arg_combine(wb, wbv, red_b[w], red_bv[w]);
    a.out[row] = wbv == INT_MAX ? -1 : wbv;
  }
}

__global__ void philox_kernel(const uint32_t* __restrict__ ctr, const uint32_t* __restrict__ key,
                              uint32_t* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    const uint2 k = make_uint2(key[2 * i], key[2 * i + 1]);
    const uint4 r = philox4x32_10(c, k);
    out[4 * i] = r.x;
    out[4 * i + 1] = r.y;
    out[4 * i + 2] = r.z;
    out[4 * i + 3] = r.w;
  }
}

// ------------------------------------------------------------------- host

int num_sms() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
  }();
  return n;
}

int elt_bytes(lp_dtype dt) { return dt == LP_F32 ? 4 : 2; }

// Tokens per tile for a launch of nrows rows: the longest tile that still
// gives kTileTarget tiles (enough for every CTA of the grid to take two), down
// to the shortest.  It does not depend on the device, so the workspace size can
// follow it exactly.
// Float32 tiles are at most 32 KB: a tile's compaction buffer holds 2048
// float32 entries, and a wide top-p window (top_p 0.99) puts about a sixth of
// a row's tokens in it.
int64_t tile_bytes_max(int eb) { return kTileBytesMax; }
int64_t tile_tokens(int eb, int64_t nrows, int64_t V) {
  int64_t tile = tile_bytes_max(eb) / eb;
  while (tile > kTileBytesMin / eb && nrows * std::max<int64_t>(1, (V + tile - 1) / tile) <
                                          kTileTarget)
    tile /= 2;
  return tile;
}
int64_t tiles_per_row(int64_t tile, int64_t V) {
  return std::max<int64_t>(1, (V + tile - 1) / tile);
}

// Workspace layout for a call of B rows of V tokens: rows per launch, tiles per
// launch at most, and the offsets of the tile summaries, the tiles' slots and
// the pool.
struct WsPlan {
  int64_t rows, tiles, pool;
  int64_t ts_off, sv_off, si_off, pv_off, pi_off, bytes;
};

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

WsPlan ws_plan(lp_dtype dt, int64_t B, int64_t V) {
  WsPlan p{};
  const int eb = elt_bytes(dt);
  const int64_t tpr_max = tiles_per_row(kTileBytesMin / eb, V);
  p.rows = std::max<int64_t>(1, std::min({B, kMaxRowsPerLaunch, kMaxTileSums / tpr_max}));
  // Tiles of one launch: at most nrows * ceil(V / longest tile) when the longest
  // tile already gives kTileTarget tiles; else tile_tokens halved the tile from
  // a length that gave fewer than kTileTarget, so at most 2 (kTileTarget - 1).
  // The bound (and the pool) grow with B and V, so a workspace sized for one
  // shape serves every smaller one.
  const int64_t rows_cap = std::min(B, kMaxRowsPerLaunch);
  p.tiles = std::max(2 * (kTileTarget - 1), rows_cap * tiles_per_row(tile_bytes_max(eb) / eb, V));
  p.pool = std::min(std::max(rows_cap * kPoolPerRow, kPoolMin), kPoolMax);
  // The header and the per-row keys must be zero when a call starts; they sit
  // in a region of fixed size at the front, which no call of any shape uses for
  // anything else, and every call leaves them zero.
  p.ts_off = int64_t(sizeof(WsHeader)) + 4 * kMaxRowsPerLaunch;
  p.sv_off = round_up(p.ts_off + p.tiles * int64_t(sizeof(TileSum)), 256);
  p.si_off = round_up(p.sv_off + p.tiles * kSlotCap * 4, 256);
  p.pv_off = round_up(p.si_off + p.tiles * kSlotCap * 4, 256);
  p.pi_off = round_up(p.pv_off + p.pool * 4, 256);
  p.bytes = round_up(p.pi_off + p.pool * 4, 256);
  return p;
}

template <int DT>
int resident_ctas() {
  static int n = [] {
    int per_sm = 0;
    if (cudaFuncSetAttribute(sample_stream_kernel<DT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_stream_kernel<DT>, kThreads,
                                                      size_t(kSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(sample_finish_kernel<DT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFinishSmem) != cudaSuccess ||
        per_sm <= 0) {
      (void)cudaGetLastError();
      per_sm = 1;
    }
    return per_sm * num_sms();
  }();
  return n;
}

template <int DT>
cudaError_t launch_sample(SampleArgs a, const WsPlan& plan, int64_t B, char* ws,
                          cudaStream_t s) {
  static std::mutex mu;
  int G;
  {
    std::lock_guard<std::mutex> lock(mu);
    G = resident_ctas<DT>();
  }
  const int eb = DT == LP_F32 ? 4 : 2;
  a.hdr = reinterpret_cast<WsHeader*>(ws);
  a.rowkey = reinterpret_cast<unsigned*>(ws + sizeof(WsHeader));
  a.ts = reinterpret_cast<TileSum*>(ws + plan.ts_off);
  a.slot_val = reinterpret_cast<float*>(ws + plan.sv_off);
  a.slot_idx = reinterpret_cast<int*>(ws + plan.si_off);
  a.pool_val = reinterpret_cast<float*>(ws + plan.pv_off);
  a.pool_idx = reinterpret_cast<int*>(ws + plan.pi_off);
  a.pool_cap = unsigned(plan.pool);
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  for (int64_t r0 = 0; r0 < B; r0 += plan.rows) {
    const int64_t nr = std::min(plan.rows, B - r0);
    const int64_t tile = tile_tokens(eb, nr, a.V);
    a.row0 = int(r0);
    a.nrows = int(nr);
    a.chunk = int(tile);
    a.tpr = int(tiles_per_row(tile, a.V));
    a.ntiles = nr * a.tpr;
    if (a.ntiles > plan.tiles) return cudaErrorInvalidValue;  // the plan bounds every launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(std::min<int64_t>(a.ntiles, G)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(kSmem);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sample_stream_kernel<DT>, a);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(unsigned(nr));
    cfg.dynamicSmemBytes = size_t(kFinishSmem);
    e = cudaLaunchKernelEx(&cfg, sample_finish_kernel<DT>, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

lp_status run_sample(const void* logits, lp_dtype dt, int64_t B, int64_t vocab,
                     int64_t logits_stride, const int32_t* bitmask, int64_t bitmask_rows,
                     int64_t bitmask_stride, const int32_t* indices, int64_t num_indices,
                     const lp_sampling_params* params, int64_t* out_ids, void* workspace,
                     int64_t workspace_bytes, cudaStream_t stream, int64_t rows_per_slot = 1,
                     const uint64_t* seeds = nullptr) {
  if (B == 0) return LP_OK;
  if (logits == nullptr && vocab > 0) return LP_ERR_INVALID_ARGUMENT;
  if (out_ids == nullptr || params == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (B > (int64_t(1) << 27) || vocab > 0x7fffffff - 64 || num_indices > 0x7fffffff)
    return LP_ERR_TOO_LARGE;
  const WsPlan plan = ws_plan(dt, B, vocab);
  if (workspace == nullptr || workspace_bytes < plan.bytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return LP_ERR_INVALID_ARGUMENT;
  const int eb = elt_bytes(dt);
  SampleArgs a{};
  a.logits = static_cast<const char*>(logits);
  a.stride_bytes = logits_stride * eb;
  a.V = int(vocab);
  a.bitmask = reinterpret_cast<const uint32_t*>(bitmask);
  a.bm_stride = bitmask_stride;
  a.bm_rows = bitmask_rows;
  a.indices = indices;
  a.n_indices = int(num_indices);
  a.temp = params->temperature;
  a.temp_s = params->temperature_scalar;
  a.topk = params->top_k;
  a.topk_s = params->top_k_scalar;
  a.topp = params->top_p;
  a.topp_s = params->top_p_scalar;
  a.minp = params->min_p;
  a.minp_s = params->min_p_scalar;
  a.seed = params->seed;
  a.offset = params->offset;
  a.rps = int(rows_per_slot);
  a.seeds = seeds;
  a.out = out_ids;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e;
  switch (dt) {
    case LP_F32: e = launch_sample<LP_F32>(a, plan, B, ws, stream); break;
    case LP_F16: e = launch_sample<LP_F16>(a, plan, B, ws, stream); break;
    default: e = launch_sample<LP_BF16>(a, plan, B, ws, stream); break;
  }
  return e == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

}  // namespace
}  // namespace lp

using namespace lp;

extern "C" int64_t lp_sample_workspace_bytes(lp_dtype dt, int64_t B, int64_t vocab_size) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16) || B < 0 || vocab_size < 0) return -1;
  if (B == 0) return 0;
  return ws_plan(dt, B, vocab_size).bytes;
}

extern "C" lp_status lp_sample(const void* logits, lp_dtype dt, int64_t B, int64_t vocab_size,
                               int64_t logits_stride, const lp_sampling_params* params,
                               int64_t* out_ids, void* workspace, int64_t workspace_bytes,
                               cudaStream_t stream) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16)) return LP_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || vocab_size < 0 || logits_stride < vocab_size) return LP_ERR_INVALID_ARGUMENT;
  return run_sample(logits, dt, B, vocab_size, logits_stride, nullptr, 0, 0, nullptr, 0, params,
                    out_ids, workspace, workspace_bytes, stream);
}

namespace {
lp_status mask_and_sample(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                          int64_t logits_stride, const int32_t* bitmask, int64_t bitmask_rows,
                          int64_t bitmask_words, int64_t bitmask_stride, int64_t vocab_size,
                          const int32_t* indices, int64_t num_indices,
                          const lp_sampling_params* params, int64_t* out_ids, void* workspace,
                          int64_t workspace_bytes, cudaStream_t stream, int64_t rows_per_slot,
                          const uint64_t* seeds) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16)) return LP_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || cols < 0 || logits_stride < cols || num_indices < 0 ||
      (num_indices > 0 && indices == nullptr))
    return LP_ERR_INVALID_ARGUMENT;
  if (bitmask == nullptr) {
    const int64_t vocab = vocab_size < 0 ? cols : vocab_size;
    if (vocab > cols) return LP_ERR_INVALID_ARGUMENT;
    return run_sample(logits, dt, B, vocab, logits_stride, nullptr, 0, 0, nullptr, 0, params,
                      out_ids, workspace, workspace_bytes, stream, rows_per_slot, seeds);
  }
  if (bitmask_words < 0 || bitmask_stride < bitmask_words || bitmask_rows < 0)
    return LP_ERR_INVALID_ARGUMENT;
  const int64_t capw = bitmask_words * 32;
  const int64_t vocab = vocab_size < 0 ? std::min(cols, capw) : vocab_size;
  if (vocab > cols || vocab > capw) return LP_ERR_INVALID_ARGUMENT;
  if (indices == nullptr && bitmask_rows < B) return LP_ERR_INVALID_ARGUMENT;
  const bool any_masked = indices == nullptr || num_indices > 0;
  return run_sample(logits, dt, B, vocab, logits_stride, any_masked ? bitmask : nullptr,
                    bitmask_rows, bitmask_stride, indices, num_indices, params, out_ids,
                    workspace, workspace_bytes, stream, rows_per_slot, seeds);
}
}  // namespace

extern "C" lp_status lp_mask_and_sample(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                        int64_t logits_stride, const int32_t* bitmask,
                                        int64_t bitmask_rows, int64_t bitmask_words,
                                        int64_t bitmask_stride, int64_t vocab_size,
                                        const int32_t* indices, int64_t num_indices,
                                        const lp_sampling_params* params, int64_t* out_ids,
                                        void* workspace, int64_t workspace_bytes,
                                        cudaStream_t stream) {
  return mask_and_sample(logits, dt, B, cols, logits_stride, bitmask, bitmask_rows,
                         bitmask_words, bitmask_stride, vocab_size, indices, num_indices, params,
                         out_ids, workspace, workspace_bytes, stream, 1, nullptr);
}

extern "C" lp_status lp_mask_and_sample_slots(const void* logits, lp_dtype dt, int64_t B,
                                              int64_t cols, int64_t logits_stride,
                                              const int32_t* bitmask, int64_t bitmask_rows,
                                              int64_t bitmask_words, int64_t bitmask_stride,
                                              int64_t vocab_size, const int32_t* indices,
                                              int64_t num_indices,
                                              const lp_sampling_params* params,
                                              int64_t rows_per_slot, const uint64_t* seeds,
                                              int64_t* out_ids, void* workspace,
                                              int64_t workspace_bytes, cudaStream_t stream) {
  if (rows_per_slot < 1 || rows_per_slot > 0x7fffffff || (B > 0 && B % rows_per_slot != 0))
    return LP_ERR_INVALID_ARGUMENT;
  return mask_and_sample(logits, dt, B, cols, logits_stride, bitmask, bitmask_rows,
                         bitmask_words, bitmask_stride, vocab_size, indices, num_indices, params,
                         out_ids, workspace, workspace_bytes, stream, rows_per_slot, seeds);
}

// Device scratch of the module itself, for callers that cannot allocate a
// workspace: zero when the module loads (the state the sampler needs), and kept
// so by every call.  Every device that loads the library holds it until exit.
namespace lp {
namespace {
constexpr int64_t kNoAllocBytes = int64_t(128) << 20;
__device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

// The array's device address on the current device, looked up once per device
// (the first call on a device does it) and then reused.
constexpr int kMaxDevices = 64;
void* noalloc_scratch(lp_status& st) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    st = LP_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess) {
      (void)cudaGetLastError();
      st = LP_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}
}  // namespace
}  // namespace lp

extern "C" lp_status lp_mask_and_sample_noalloc(const void* logits, lp_dtype dt, int64_t B,
                                                int64_t cols, int64_t logits_stride,
                                                const int32_t* bitmask, int64_t bitmask_rows,
                                                int64_t bitmask_words, int64_t bitmask_stride,
                                                int64_t vocab_size, const int32_t* indices,
                                                int64_t num_indices,
                                                const lp_sampling_params* params,
                                                int64_t* out_ids, cudaStream_t stream) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16)) return LP_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || cols < 0 || bitmask_words < 0) return LP_ERR_INVALID_ARGUMENT;
  if (B == 0) return LP_OK;
  // the vocabulary the call resolves to (as lp_mask_and_sample resolves it) sizes
  // the scratch; an inconsistent one is refused by that entry point below
  int64_t vocab = vocab_size >= 0 ? vocab_size
                  : bitmask != nullptr ? std::min(cols, bitmask_words * 32)
                                       : cols;
  vocab = std::min(std::max<int64_t>(vocab, 0), cols);
  const int64_t need = lp_sample_workspace_bytes(dt, B, vocab);
  if (need < 0 || need > kNoAllocBytes) return LP_ERR_TOO_LARGE;
  lp_status st = LP_OK;
  void* ws = noalloc_scratch(st);
  if (ws == nullptr) return st;
  return lp_mask_and_sample(logits, dt, B, cols, logits_stride, bitmask, bitmask_rows,
                            bitmask_words, bitmask_stride, vocab_size, indices, num_indices,
                            params, out_ids, ws, kNoAllocBytes, stream);
}

extern "C" lp_status lp_philox4x32_10(const uint32_t* counters, const uint32_t* keys,
                                      uint32_t* out, int64_t n, cudaStream_t stream) {
  if (n < 0) return LP_ERR_INVALID_ARGUMENT;
  if (n == 0) return LP_OK;
  if (!counters || !keys || !out) return LP_ERR_INVALID_ARGUMENT;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  philox_kernel<<<unsigned(blocks), 256, 0, stream>>>(counters, keys, out, n);
  return cudaGetLastError() == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

extern "C" const char* lp_status_string(lp_status status) {
  switch (status) {
    case LP_OK: return "ok";
    case LP_ERR_INVALID_ARGUMENT: return "invalid argument";
    case LP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case LP_ERR_CUDA: return "CUDA launch failed";
    case LP_ERR_TOO_LARGE:
      return "size too large: past the kernels' 32-bit index range, or (noalloc) past the "
             "library's fixed device scratch";
    default: return "unknown status";
  }
}
