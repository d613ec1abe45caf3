// sample.cu -- fused bitmask + temperature + top-k ∩ top-p ∩ min-p + Gumbel-max
// sampler (Kernel Hub "logits-processor", Ops "sample" and "How it works";
// unsatisfiable rows as in TensorRT-Edge-LLM "Guided Decoder").
//
// GB300 design: one streaming pass over HBM through the Tensor Memory
// Accelerator, in a persistent grid.  A row is split over a thread-block cluster
// of S CTAs; the resident clusters take the rows round-robin.  Each CTA streams
// its parts of its rows through a ring of four 8 KB shared-memory stages: one
// thread keeps bulk copies (cp.async.bulk, with the stage's bitmask words) in
// flight on mbarriers, running up to one row ahead, so the next row's loads
// overlap this row's reductions; the 256 threads consume each landed stage from
// shared memory.  The CTAs of a row combine partial results through distributed
// shared memory (DSMEM) behind cluster barriers; nothing is written to global
// memory but the ids.
//
// Per row, in the stream:
//   * candidate max, the vector holding it (its lowest index is found after the
//     pass), the candidate count and, for top-p rows, an online softmax sum;
//   * filtered rows: every candidate within a window below the running maximum
//     (shared by the CTA's warps through a shared-memory atomicMax) is appended
//     to a compaction buffer.  The window is exactly the min-p bound when min-p is
//     on (max + T ln min_p); otherwise a number of temperature units growing with
//     ln(1 / (1 - top_p)) for top-p and a fixed number of logits for top-k.  The
//     running maximum never exceeds the row maximum, so the buffer holds every
//     candidate in [max - window, max];
//   * rows without filters draw Gumbel-max directly (no threshold needed),
//     skipping any token whose best possible score is below the running best.
// After the stream (one exchange): no candidate -> -1; greedy -> argmax;
// unfiltered -> the best score's token.  Filtered rows find the keep-threshold
// max(t_k, t_p, t_m) by an MSD radix select over the order-preserving key of the
// logit -- counts for top-k and 2^-40 fixed-point softmax mass for top-p, pre-summed
// per warp (match_any + redux) and summed over the cluster per digit; one descent
// serves both filters: the threshold is the largest key at which "count >= k" or
// "mass >= top_p S" first holds.  The descent runs on the buffer, counting only the
// region where the buffer is complete; if the threshold is not found there (or a
// buffer overflowed) the CTAs stream their parts again (an L2 hit in practice) and
// select and draw from those.  The draw is Gumbel-max over the kept set with
// Philox4x32-10 noise keyed by (seed, row, offset).
// Masses are integers, so every cluster-wide sum is exact and order-independent;
// the softmax sum is reduced in a fixed order.  Results are deterministic in
// (seed, offset).
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <map>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace lp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRing = 4;                 // stages in flight per CTA
constexpr int kPieceBytes = 8192;        // bytes of logits per stage
constexpr int kPieceWords = kPieceBytes / 2 / 32 + 2;  // bitmask words a stage can need
constexpr int kMaskSlot = (16 + 4 * kPieceWords + 15) / 16 * 16;
constexpr int kPerPiece = kPieceBytes / 16 / 256;  // vectors of a piece per thread
constexpr int kKBins = 128;              // log-spaced bins of (row max - thread max)
constexpr int kKBase = (127 - 6) << 3;   // code of 2^-6 (8 exponent + 3 fraction bits)
constexpr int kMaxSplit = 16;
constexpr int kCap = 3072;               // compaction entries per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kWindowK = 6.f;          // top-k window, in logits
constexpr int kSmem = kRing * kPieceBytes + kRing * kMaskSlot + kCap * 8;
constexpr uint32_t kMaxWaitTries = 1u << 22;

struct SampleArgs {
  const char* logits;
  int64_t stride_bytes;
  int B;
  int V;
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
  int64_t* out;
  int chunk;  // tokens per CTA (a multiple of 32)
  int ncl;    // clusters in the grid; cluster c owns rows c, c + ncl, ...
};

struct Xchg {  // per-CTA values read by the other CTAs of the cluster
  float max;
  int arg;
  float sum;  // softmax sum relative to max
  int ncand;
  int overflow;
  int err;
  float best;
  int best_v;
};

struct Hist {  // radix histograms, double-buffered by pass parity
  unsigned long long mass[2][256];
  unsigned cnt[2][256];
};

__device__ __forceinline__ void arg_combine(float& s, int& v, float s2, int v2) {
  if (s2 > s || (s2 == s && v2 < v)) {
    s = s2;
    v = v2;
  }
}

// Merge two partial row summaries (max, lowest index of the max and -- when
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

// Log-spaced bin of d >= 0: bin 0 holds d < 2^-6, then 8 bins per octave; the
// last bin also takes everything larger.
__device__ __forceinline__ int kbin(float d) {
  const int code = int(__float_as_uint(d) >> 20);
  return min(max(code - kKBase + 1, 0), kKBins - 1);
}
// Exclusive upper edge of bin j (j < kKBins - 1).
__device__ __forceinline__ float kbin_hi(int j) {
  return j == 0 ? 0.015625f : __uint_as_float(unsigned(j + kKBase) << 20);
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
// Bounded wait for the phase of the given parity to complete.  Each try_wait
// suspends the thread for a hardware-chosen time slice; after kMaxWaitTries
// failures (far beyond any copy's latency) it gives up and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity) {
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

// ------------------------------------------------------------ row part

// One CTA's part of one row: local element i is token start + i, at byte
// mis + i * EB of a 16-byte aligned window starting at g0.  The window is
// streamed in pieces of kPieceBytes.  Whole 16-byte vectors [qf0, qf1) of the
// window arrive by bulk copy; the ragged first and last vectors are read from
// global memory when used.  Each piece's bitmask words arrive with it: words
// [m_lo, m_hi) (relative to the part) sit at byte mmis + 4 (w - m_lo) of the
// piece's mask slot; other words are read from global memory.
template <int DT>
struct Part {
  using E = Elt<DT>;
  static constexpr int EPV = E::kPerVec;
  static constexpr int EB = E::kBytes;
  static constexpr uint32_t ALL = (1u << EPV) - 1u;
  const char* g0;
  const uint32_t* gmask;  // the part's bitmask words (masked rows)
  int start, n_local, mis, win, nvec, nwords, qf0, qf1, npieces;
  bool masked;

  __device__ __forceinline__ void init(const SampleArgs& a, int row, int rank, bool m) {
    start = rank * a.chunk;
    n_local = max(0, min(a.chunk, a.V - start));
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
  // the 16-byte aligned interior [m_lo, m_hi) of words [w0, w1), and the byte
  // offset of word m_lo in its slot
  __device__ __forceinline__ void mask_interior(int w0, int w1, int& m_lo, int& m_hi,
                                                int& mmis) const {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(gmask + w0);
    const int lead = int(((16 - (a0 & 15)) & 15) >> 2);
    m_lo = min(w0 + lead, w1);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(gmask + w1) & ~uintptr_t(15);
    m_hi = max(m_lo, int((a1 - reinterpret_cast<uintptr_t>(gmask)) >> 2));
    mmis = 0;
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
  // candidate bits of vector q (element e a token of this part kept by the mask),
  // its mask words taken from `mw` (words [m_lo, m_hi)) or global memory
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

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) sample_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  using Pt = Part<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int kLow = int(E::kLowKeyBit);

  cg::cluster_group cluster = cg::this_cluster();
  const int C = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int cid = int(blockIdx.x) / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto xsync = [&]() {
    if (C > 1)
      cluster.sync();
    else
      __syncthreads();
  };

  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* const ring = smem;
  unsigned char* const mring = smem + kRing * kPieceBytes;
  float* const bval = reinterpret_cast<float*>(mring + kRing * kMaskSlot);
  int* const bidx = reinterpret_cast<int*>(bval + kCap);

  __shared__ Xchg xchg[2];              // by row parity: read by peers without a trailing barrier
  __shared__ float tmaxs[2][kThreads];  // per-thread maxima, by row parity
  __shared__ Hist hist;                 // by radix-pass parity
  __shared__ float red_f[kWarps], red_s[kWarps], red_b[kWarps];
  __shared__ int red_i[kWarps], red_n[kWarps], red_bv[kWarps];
  __shared__ unsigned scan_c[kWarps];
  __shared__ unsigned long long scan_m[kWarps];
  __shared__ unsigned kmerge[kKBins];
  __shared__ int s_count, s_sel, s_err, s_i[4];
  __shared__ float s_f[3];
  __shared__ unsigned s_runkey, s_above_c;
  __shared__ unsigned long long s_above_m;
  __shared__ int s_masked[2];  // masked flag of the row of each parity
  __shared__ __align__(8) uint64_t full[kRing];
  __shared__ uint4 keep_tab[256];  // 16-bit types: per-word keep masks of 8 element bits
  __shared__ int4 pmeta[kRing];  // per slot: vectors [x, y), staged mask words [z, w)
  __shared__ int pwhole[kRing];  // per slot: every vector of the piece is a whole vector

  if (tid == 0) {
    s_err = 0;
    for (int r = 0; r < kRing; ++r) mbar_init(&full[r], 1);
    mbar_init_fence();
  }
  keep_tab[tid] = make_uint4(keep_mask16(tid, 0), keep_mask16(tid, 1), keep_mask16(tid, 2),
                             keep_mask16(tid, 3));
  __syncthreads();

  const uint2 key = make_uint2(uint32_t(a.seed), uint32_t(a.seed >> 32));
  auto row_of = [&](int it) { return cid + it * a.ncl; };
  auto masked_of = [&](int row) -> bool {  // block-uniform
    if (!a.bitmask) return false;
    if (a.indices == nullptr) return true;
    int found = 0;
    for (int i = tid; i < a.n_indices; i += kThreads) found |= (a.indices[i] == row);
    return __syncthreads_or(found) != 0 && row < a.bm_rows;
  };

  // ---------------------------------------------------------------- the ring
  // Pieces of this CTA's rows are copied in row order into slot (n % kRing) of
  // the n-th piece; thread 0 keeps up to kRing of them in flight, at most one
  // row ahead of the row being consumed, so the next row's loads overlap this
  // row's reductions.
  uint32_t issued = 0, consumed = 0, lost = 0;
  int p_iter = 0, p_piece = 0;  // producer position (thread 0)
  auto issue = [&](const Pt& g, int j) {
    const int slot = int(issued % kRing);
    ++issued;
    int q0, q1;
    g.piece_vecs(j, q0, q1);
    const int v0 = max(q0, g.qf0), v1 = min(q1, g.qf1);
    const uint32_t vbytes = v1 > v0 ? uint32_t(16 * (v1 - v0)) : 0u;
    uint32_t mbytes = 0;
    int w0 = 0, w1 = 0, m_lo = 0, m_hi = 0, mmis = 0;
    if (g.masked) {
      g.piece_words(j, w0, w1);
      g.mask_interior(w0, w1, m_lo, m_hi, mmis);
      mbytes = uint32_t(4 * (m_hi - m_lo));
    }
    pmeta[slot] = make_int4(q0, q1, m_lo, m_hi);  // published by the arrive below
    pwhole[slot] = q0 >= g.qf0 && q1 <= g.qf1;
    if (s_err) {  // a copy went missing earlier: start no more (rows report -2)
      mbar_expect_tx(&full[slot], 0);
      return;
    }
    mbar_expect_tx(&full[slot], vbytes + mbytes);
    if (vbytes)
      bulk_load(ring + slot * kPieceBytes + 16 * (v0 - q0), g.g0 + 16 * v0, vbytes, &full[slot]);
    if (mbytes) bulk_load(mring + slot * kMaskSlot, g.gmask + m_lo, mbytes, &full[slot]);
  };
  __shared__ Pt pg;  // producer: geometry of row p_iter (thread 0 only)
  int pg_iter = -1;  // the iteration pg describes
  auto top_up = [&](int cur) {  // thread 0 only
    while (issued - consumed < uint32_t(kRing)) {
      const int prow = row_of(p_iter);
      if (prow >= a.B || p_iter > cur + 1) break;
      if (pg_iter != p_iter) {
        pg.init(a, prow, rank, s_masked[p_iter & 1] != 0);
        pg_iter = p_iter;
      }
      if (p_piece < pg.npieces) {
        issue(pg, p_piece);
        ++p_piece;
      } else {
        ++p_iter;
        p_piece = 0;
      }
    }
  };

  if (row_of(0) < a.B) {
    const bool m0 = masked_of(row_of(0));
    if (tid == 0) s_masked[0] = m0;
  }
  int npass = 0;  // radix passes so far: histogram parity

  for (int it = 0; row_of(it) < a.B; ++it) {
    const int row = row_of(it);
    const int par = it & 1;
    __syncthreads();  // the previous row is done in this CTA
    if (row_of(it + 1) < a.B) {
      const bool mn = masked_of(row_of(it + 1));
      if (tid == 0) s_masked[par ^ 1] = mn;
    }
    if (tid == 0) {
      s_count = 0;
      s_runkey = fkey(-INFINITY);
    }
    if (tid < kKBins) kmerge[tid] = 0u;
    __syncthreads();
    if (tid == 0) top_up(it);

    Pt pt;
    pt.init(a, row, rank, s_masked[par] != 0);
    const float T = a.temp ? a.temp[row] : a.temp_s;
    int k = a.topk ? a.topk[row] : a.topk_s;
    const float tp = a.topp ? a.topp[row] : a.topp_s;
    const float mp = a.minp ? a.minp[row] : a.minp_s;
    const bool greedy = !(T > 0.f) || k == 1;
    const bool has_p = !greedy && tp < 1.f;
    const bool has_m = !greedy && mp > 0.f;
    const bool has_k0 = !greedy && k > 0;
    const bool unfiltered = !greedy && !has_p && !has_m && !has_k0;
    const bool compact = !greedy && !unfiltered;
    const float c2 = greedy ? 0.f : kLog2e / T;
    const float tl = has_m ? T * logf(mp) : 0.f;  // min-p bound below the maximum: max + tl
    float delta = INFINITY;                       // compaction window below the running max
    if (has_m) delta = fminf(delta, -tl);
    if (has_p) delta = fminf(delta, T * (2.f + 2.5f * logf(1.f / fmaxf(1.f - tp, 1e-6f))));
    if (has_k0) delta = fminf(delta, kWindowK);
    if (!(delta > 0.f)) delta = 0.f;

    // Gumbel score of candidate (z = x / T, token v); w4/wgrp cache v's Philox block
    auto score_of = [&](float z, int v, uint4& w4, int& wgrp) {
      const int grp = v >> 2;
      if (grp != wgrp) {
        w4 = philox4x32_10(make_uint4(uint32_t(grp), uint32_t(row), uint32_t(a.offset),
                                      uint32_t(a.offset >> 32)),
                           key);
        wgrp = grp;
      }
      const uint32_t word = (v & 3) == 0 ? w4.x : (v & 3) == 1 ? w4.y : (v & 3) == 2 ? w4.z : w4.w;
      return z + gumbel_from_word(word);
    };

    // ------------------------------------------------- stream the row part
    float m = -INFINITY, sm = 0.f;  // running max and softmax sum relative to it
    int mq = -1, cnt = 0;           // vector of the running max; candidate bits seen
    float best = -INFINITY;         // unfiltered rows: running best score
    int bestv = INT_MAX;
    uint4 w4 = make_uint4(0, 0, 0, 0);
    int wgrp = -1;
    bool stream_ok = true;
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
      const bool whole = pwhole[slot] != 0;
      const unsigned char* data = ring + slot * kPieceBytes;
      const uint32_t* mw = reinterpret_cast<const uint32_t*>(mring + slot * kMaskSlot);
      // vector q of this piece, its candidate bits, and (16-bit types) the vector
      // with every non-candidate element replaced by -inf
      auto load = [&](int q, uint4& raw, uint32_t& cb) {
        const bool staged = whole || (q >= pt.qf0 && q < pt.qf1);
        raw = staged ? *reinterpret_cast<const uint4*>(data + 16 * (q - pm.x)) : pt.gvec(q);
        int i0;
        cb = (whole && !pt.masked) ? Pt::ALL : pt.bits(q, i0, mw, pm.z, pm.w);
      };
      auto masked_vec = [&](const uint4& raw, uint32_t cb) -> uint4 {
        if (cb == Pt::ALL) return raw;
        if (Pt::EB == 4) {
          constexpr uint32_t kNegInf = 0xff800000u;
          return make_uint4((cb & 1u) ? raw.x : kNegInf, (cb & 2u) ? raw.y : kNegInf,
                            (cb & 4u) ? raw.z : kNegInf, (cb & 8u) ? raw.w : kNegInf);
        }
        const uint32_t ninf2 = DT == LP_BF16 ? 0xff80ff80u : 0xfc00fc00u;
        const uint4 t = keep_tab[cb];
        return make_uint4((raw.x & t.x) | (ninf2 & ~t.x), (raw.y & t.y) | (ninf2 & ~t.y),
                          (raw.z & t.z) | (ninf2 & ~t.z), (raw.w & t.w) | (ninf2 & ~t.w));
      };
      float vms[kPerPiece];
#pragma unroll
      for (int r = 0; r < kPerPiece; ++r) {
        const int q = pm.x + r * kThreads + tid;
        vms[r] = -INFINITY;
        if (q >= pm.y) continue;
        uint4 raw;
        uint32_t cb;
        load(q, raw, cb);
        if (!cb) continue;
        const uint4 mv = masked_vec(raw, cb);
        const float vm = VecMax<DT>::run(mv, Pt::ALL);
        vms[r] = vm;
        cnt += __popc(cb);
        if (vm > m) {
          if (has_p) sm *= ex2((m - vm) * c2);  // 0 while m is still -inf
          m = vm;
          mq = q;
        }
        if (has_p && vm > -INFINITY) {  // m is finite: -inf elements add 0
          const float off = m * c2;
#pragma unroll
          for (int e = 0; e < EPV; ++e) sm += ex2(fmaf(E::get(mv, e), c2, -off));
        }
        if (unfiltered) {
          const int i0 = (16 * q - pt.mis) / Pt::EB;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float x = E::get(mv, e);
            if (!(x > -INFINITY)) continue;
            const float z = __fdiv_rn(x, T);
            if (z + kGumbelMax < best) continue;  // cannot win
            const int v = pt.start + i0 + e;
            arg_combine(best, bestv, score_of(z, v, w4, wgrp), v);
          }
        }
      }
      if (compact) {  // warp-uniform: append the piece's candidates within the window
        float wm = m;
#pragma unroll
        for (int o = 16; o; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFullWarp, wm, o));
        if (lane == 0 && wm > -INFINITY) atomicMax(&s_runkey, fkey(wm));
        const float rm = fmaxf(wm, key_float(*(volatile unsigned*)&s_runkey));
        const float cut = __fsub_rd(rm, delta);
#pragma unroll
        for (int r = 0; r < kPerPiece; ++r) {
          // a lane without a vector has vms = -inf, which must not pass a cut of -inf
          const bool live = vms[r] > -INFINITY && vms[r] >= cut;
          if (!__any_sync(kFullWarp, live)) continue;
          const int q = pm.x + r * kThreads + tid;
          uint32_t pass = 0;
          uint4 raw = make_uint4(0, 0, 0, 0);
          if (live) {
            uint32_t cb;
            load(q, raw, cb);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const float x = E::get(raw, e);
              if (((cb >> e) & 1u) && x >= cut && x > -INFINITY) pass |= 1u << e;
            }
          }
          const int n = __popc(pass);
          int incl = n;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullWarp, incl, o);
            if (lane >= o) incl += y;
          }
          int pos = 0;
          if (lane == 31) pos = atomicAdd(&s_count, incl);
          pos = __shfl_sync(kFullWarp, pos, 31) + incl - n;
          const int i0 = (16 * q - pt.mis) / Pt::EB;
          while (pass) {
            const int e = __ffs(pass) - 1;
            pass &= pass - 1;
            if (pos < kCap) {
              bval[pos] = E::get(raw, e);
              bidx[pos] = pt.start + i0 + e;
            }
            ++pos;
          }
        }
      }
      __syncthreads();  // every thread is done with the slot
      if (tid == 0) top_up(it);
    }

    // -------------------------------------------------------- row summaries
    tmaxs[par][tid] = m;
    int targ = INT_MAX;
    if (mq >= 0) {  // lowest index of the thread's maximum, in the first vector holding it
      int i0;
      const uint32_t cb = pt.bits(mq, i0, nullptr, 0, 0);
      const uint4 raw = pt.gvec(mq);
#pragma unroll
      for (int e = EPV - 1; e >= 0; --e)
        if (((cb >> e) & 1u) && E::get(raw, e) == m) targ = pt.start + i0 + e;
    }
    {
      float wm = m, ws = sm, wb = best;
      int wv = targ, wn = cnt, wbv = bestv;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFullWarp, wm, o);
        const float s2 = __shfl_xor_sync(kFullWarp, ws, o);
        const int v2 = __shfl_xor_sync(kFullWarp, wv, o);
        wn += __shfl_xor_sync(kFullWarp, wn, o);
        row_combine(wm, wv, ws, m2, v2, s2, c2, has_p);
        if (unfiltered) {
          const float b2 = __shfl_xor_sync(kFullWarp, wb, o);
          const int bv2 = __shfl_xor_sync(kFullWarp, wbv, o);
          arg_combine(wb, wbv, b2, bv2);
        }
      }
      if (lane == 0) {
        red_f[warp] = wm;
        red_s[warp] = ws;
        red_i[warp] = wv;
        red_n[warp] = wn;
        red_b[warp] = wb;
        red_bv[warp] = wbv;
      }
    }
    const int cta_err = __syncthreads_or(!stream_ok || s_err != 0);
    if (warp == 0) {
      float wm = -INFINITY, ws = 0.f, wb = -INFINITY;
      int wv = INT_MAX, wn = 0, wbv = INT_MAX;
      if (lane < kWarps) {
        wm = red_f[lane];
        ws = red_s[lane];
        wv = red_i[lane];
        wn = red_n[lane];
        wb = red_b[lane];
        wbv = red_bv[lane];
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
      if (lane == 0) {
        Xchg& x = xchg[par];
        x.max = wm;
        x.arg = wv;
        x.sum = ws;
        x.ncand = wn;
        x.best = wb;
        x.best_v = wbv;
        x.overflow = s_count > kCap;
        x.err = cta_err;
      }
    }
    xsync();  // #1: every CTA's summary is visible to its cluster
    if (warp == 0) {
      float wm = -INFINITY, ws = 0.f, wb = -INFINITY;
      int wv = INT_MAX, wn = 0, wbv = INT_MAX, ov = 0, er = 0;
      if (lane < C) {
        const Xchg* p = cluster.map_shared_rank(&xchg[par], lane);
        wm = p->max;
        wv = p->arg;
        ws = p->sum;
        wn = p->ncand;
        wb = p->best;
        wbv = p->best_v;
        ov = p->overflow;
        er = p->err;
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
      }
      ov = __any_sync(kFullWarp, ov != 0);
      er = __any_sync(kFullWarp, er != 0);
      if (lane == 0) {
        s_f[0] = wm;
        s_f[1] = ws;
        s_i[0] = wv;
        s_i[1] = wn;
        s_i[2] = wbv;
        s_i[3] = ov | (er << 1);
      }
    }
    __syncthreads();
    const float lmax = s_f[0];
    const float S = s_f[1];
    const int larg = s_i[0];
    const int ncand_ub = s_i[1];  // candidates counted by their bits (-inf included)
    const bool row_err = (s_i[3] >> 1) != 0;

    if (row_err || lmax == -INFINITY || greedy || unfiltered) {
      if (rank == 0 && tid == 0)
        a.out[row] = row_err ? -2
                     : lmax == -INFINITY ? -1
                     : greedy ? larg
                              : (s_i[2] == INT_MAX ? -1 : s_i[2]);
      continue;
    }
    const bool any_overflow = (s_i[3] & 1) != 0;
    const int nbuf = min(s_count, kCap);

    // ------------------------------------------------------- filter bounds
    if (k > 0 && k >= ncand_ub) k = 0;  // keeps every candidate
    const bool has_k = k > 0;
    const float fm = has_m ? fminf(__fadd_ru(lmax, tl), lmax) : -INFINITY;
    // top-k: the k-th largest per-thread maximum of the cluster bounds t_k from below
    int jk = -1;
    if (has_k && !has_m && k <= C * kThreads) {
      for (int r = 0; r < C; ++r) {
        const float v = cluster.map_shared_rank(&tmaxs[par][0], r)[tid];
        if (v > -INFINITY) atomicAdd(&kmerge[kbin(lmax - v)], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        const unsigned c0 = kmerge[4 * lane], c1 = kmerge[4 * lane + 1];
        const unsigned cc2 = kmerge[4 * lane + 2], c3 = kmerge[4 * lane + 3];
        unsigned incl = c0 + c1 + cc2 + c3;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(kFullWarp, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned excl = incl - (c0 + c1 + cc2 + c3);
        const unsigned kk = unsigned(k);
        int j = -1;
        if (excl < kk && incl >= kk) {
          unsigned cum = excl + c0;
          j = cum >= kk ? 4 * lane
                        : ((cum += c1) >= kk ? 4 * lane + 1
                                             : ((cum += cc2) >= kk ? 4 * lane + 2 : 4 * lane + 3));
        }
        const unsigned found = __ballot_sync(kFullWarp, j >= 0);
        j = __shfl_sync(kFullWarp, j, found ? __ffs(found) - 1 : 0);
        if (lane == 0) s_i[2] = found ? j : -1;
      }
      __syncthreads();
      jk = s_i[2];
    }
    float fcut = fm;  // certified lower bound of the keep-threshold
    if (jk >= 0 && jk < kKBins - 1) fcut = fmaxf(fcut, __fsub_rd(lmax, kbin_hi(jk)));
    if (has_p) {
      float D = logf(float(ncand_ub) / (fmaxf(1.f - tp, 1e-30f) * S));
      D = fmaxf(D, 0.f) * 1.001f + 1e-3f;
      fcut = fmaxf(fcut, __fsub_rd(lmax, T * D));
    }
    // the buffer holds every candidate in [lo_w, lmax]
    const float lo_w = has_m ? fm : __fsub_ru(lmax, delta);

    // Re-reads this CTA's part from global memory (the ring is prefetching the
    // next row): f(raw, cb, i0) per vector, warp-uniform.
    auto reread = [&](auto&& f) {
      for (int base = 0; base < pt.nvec; base += kThreads) {
        const int q = base + tid;
        int i0 = 0;
        uint32_t cb = 0;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (q < pt.nvec) {
          cb = pt.bits(q, i0, nullptr, 0, 0);
          if (cb) raw = pt.gvec(q);
        }
        f(raw, cb, i0);
      }
    };

    // ---------------------------------- radix select of the threshold
    unsigned long long P = 0ull;  // fixed-point top-p mass target
    if (has_p) {
      const float t = fmaxf(tp, 0.f) * S * 1099511627776.0f;
      P = t >= 1.8e19f ? ~0ull : static_cast<unsigned long long>(t);
    }
    // Largest key x >= key(lo) with count(>= x) >= k (top-k) or mass(>= x) >= P
    // (top-p), counting candidates of the buffer or of a re-read of the part.
    // False when none exists.
    auto descend = [&](bool from_buffer, float lo, uint32_t& out_key) -> bool {
      const uint32_t klo = fkey(lo), khi = fkey(lmax);
      const uint32_t diff = klo ^ khi;
      int top = diff ? 32 - __clz(diff) : kLow + 1;  // one past the highest differing bit
      top = max(top, kLow + 1);
      int shift = max(top - 8, kLow);
      uint32_t prefix = top >= 32 ? 0u : khi & ~((1u << top) - 1u);
      unsigned above_c = 0;
      unsigned long long above_m = 0;
      for (;;) {
        const int hp = npass & 1;
        ++npass;
        hist.cnt[hp][tid] = 0u;
        hist.mass[hp][tid] = 0ull;
        if (tid == 0) s_sel = -1;
        __syncthreads();
        const uint32_t himask = top >= 32 ? 0u : ~((1u << top) - 1u);
        const uint32_t dmask = (1u << (top - shift)) - 1u;
        // warp-uniform: every lane calls with its element (or part = false)
        auto add = [&](float x, bool part) {
          int d = -1;
          if (part && x >= lo) {
            const uint32_t kx = fkey(x);
            if (((kx ^ prefix) & himask) == 0u) d = int((kx >> shift) & dmask);
          }
          if (!__any_sync(kFullWarp, d >= 0)) return;
          const unsigned peers = __match_any_sync(kFullWarp, d);
          if (d < 0) return;
          const bool leader = lane == __ffs(peers) - 1;
          if (has_p) {
            const float e = ex2((x - lmax) * c2);
            const unsigned long long mm = __float2ull_rn(e * 1099511627776.0f);
            const unsigned hi = __reduce_add_sync(peers, unsigned(mm >> 20));
            const unsigned lw = __reduce_add_sync(peers, unsigned(mm & 0xFFFFFu));
            if (leader)
              atomicAdd(&hist.mass[hp][d], (static_cast<unsigned long long>(hi) << 20) + lw);
          }
          if (leader) atomicAdd(&hist.cnt[hp][d], unsigned(__popc(peers)));
        };
        if (from_buffer) {
          for (int b0 = warp * 32; b0 < nbuf; b0 += kThreads) {
            const int i = b0 + lane;
            add(i < nbuf ? bval[i] : 0.f, i < nbuf);
          }
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
        xsync();
        // bin tid summed over the cluster, then a descending inclusive scan
        unsigned c = 0;
        unsigned long long mass = 0;
        for (int r = 0; r < C; ++r) {
          const Hist* h = cluster.map_shared_rank(&hist, r);
          c += h->cnt[hp][tid];
          mass += h->mass[hp][tid];
        }
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
        const bool okb = cc > 0u && ((has_k && cc >= unsigned(k)) || (has_p && cm >= P));
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

    float thr = fm;
    bool from_buffer = !any_overflow;
    const float lo_b = fmaxf(lo_w, fcut);
    if (has_k || has_p) {
      uint32_t kx = 0;
      bool found = false;
      if (from_buffer) {
        found = descend(true, lo_b, kx);
        if (!found && !(fm >= lo_b)) from_buffer = false;
      }
      if (!from_buffer) found = descend(false, fcut, kx);
      if (found) thr = fmaxf(key_float(kx), fm);
    } else if (from_buffer && !(fm >= lo_w)) {
      from_buffer = false;
    }

    // ----------------------------------------------------------------- draw
    best = -INFINITY;
    bestv = INT_MAX;
    if (from_buffer) {
      for (int i = tid; i < nbuf; i += kThreads) {
        const float x = bval[i];
        if (!(x >= thr)) continue;
        uint4 w;
        int g = -1;
        const int v = bidx[i];
        arg_combine(best, bestv, score_of(__fdiv_rn(x, T), v, w, g), v);
      }
    } else {
      wgrp = -1;
      reread([&](const uint4& raw, uint32_t cb, int i0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float x = E::get(raw, e);
          if (!((cb >> e) & 1u) || !(x >= thr) || !(x > -INFINITY)) continue;
          const float z = __fdiv_rn(x, T);
          if (z + kGumbelMax < best) continue;
          const int v = pt.start + i0 + e;
          arg_combine(best, bestv, score_of(z, v, w4, wgrp), v);
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
      xchg[par].best = wb;
      xchg[par].best_v = wbv;
    }
    xsync();
    if (rank == 0 && tid == 0) {
      float wb = -INFINITY;
      int wbv = INT_MAX;
      for (int r = 0; r < C; ++r) {
        const Xchg* p = cluster.map_shared_rank(&xchg[par], r);
        arg_combine(wb, wbv, p->best, p->best_v);
      }
      a.out[row] = wbv == INT_MAX ? -1 : wbv;
    }
  }

  // Leave only once every stage is idle and the peers are done reading this
  // CTA: a stage whose wait timed out gets one more bounded wait.
  for (int sl = 0; sl < kRing; ++sl)
    if ((lost >> sl) & 1u) (void)mbar_wait(&full[sl], (lost >> (sl + 8)) & 1u);
  if (C > 1) cluster.sync();
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

// Tokens per CTA when a row is split over S CTAs (a multiple of 32, so a CTA's
// bitmask words are its own).
int64_t chunk_for(int64_t V, int S) {
  int64_t c = (V + S - 1) / S;
  c = (c + 31) / 32 * 32;
  return std::max<int64_t>(c, 32);
}

// CTAs per row: one, unless there are fewer rows than SMs; then rows are split
// over clusters until every SM has work, keeping at least 4096 tokens per CTA.
int split_for(int64_t B, int64_t V) {
  int S = 1;
  while (S < kMaxSplit && B * S < int64_t(num_sms()) && chunk_for(V, 2 * S) >= 4096) S *= 2;
  return S;
}

template <int DT>
cudaError_t launch_sample(SampleArgs a, int64_t B, int64_t V, cudaStream_t s) {
  static std::mutex mu;
  static bool configured = false;
  static std::map<int, int> clusters;  // resident clusters by cluster size
  int S = split_for(B, V);
  int resident = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(sample_kernel<DT>,
                                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(sample_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmem);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    for (;;) {
      auto it = clusters.find(S);
      if (it == clusters.end()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(S) * 64u);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = size_t(kSmem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(S);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sample_kernel<DT>, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = 0;
        }
        it = clusters.emplace(S, n).first;
      }
      resident = it->second;
      if (resident > 0 || S == 1) break;
      S /= 2;  // this cluster shape cannot be co-scheduled: try a smaller one
    }
  }
  if (resident <= 0) resident = std::max(1, 3 * num_sms() / S);
  a.chunk = int(chunk_for(V, S));
  a.ncl = int(std::min<int64_t>(B, resident));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.ncl) * unsigned(S));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(kSmem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_kernel<DT>, a);
}

lp_status run_sample(const void* logits, lp_dtype dt, int64_t B, int64_t vocab,
                     int64_t logits_stride, const int32_t* bitmask, int64_t bitmask_rows,
                     int64_t bitmask_stride, const int32_t* indices, int64_t num_indices,
                     const lp_sampling_params* params, int64_t* out_ids, cudaStream_t stream) {
  if (B == 0) return LP_OK;
  if (logits == nullptr && vocab > 0) return LP_ERR_INVALID_ARGUMENT;
  if (out_ids == nullptr || params == nullptr) return LP_ERR_INVALID_ARGUMENT;
  if (B * int64_t(kMaxSplit) > 0x7fffffff || vocab > 0x7fffffff - 64 ||
      num_indices > 0x7fffffff)
    return LP_ERR_TOO_LARGE;
  const int eb = dt == LP_F32 ? 4 : 2;
  SampleArgs a{};
  a.logits = static_cast<const char*>(logits);
  a.stride_bytes = logits_stride * eb;
  a.B = int(B);
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
  a.out = out_ids;
  cudaError_t e;
  switch (dt) {
    case LP_F32: e = launch_sample<LP_F32>(a, B, vocab, stream); break;
    case LP_F16: e = launch_sample<LP_F16>(a, B, vocab, stream); break;
    default: e = launch_sample<LP_BF16>(a, B, vocab, stream); break;
  }
  return e == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

}  // namespace
}  // namespace lp

using namespace lp;

extern "C" lp_status lp_sample(const void* logits, lp_dtype dt, int64_t B, int64_t vocab_size,
                               int64_t logits_stride, const lp_sampling_params* params,
                               int64_t* out_ids, cudaStream_t stream) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16)) return LP_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || vocab_size < 0 || logits_stride < vocab_size) return LP_ERR_INVALID_ARGUMENT;
  return run_sample(logits, dt, B, vocab_size, logits_stride, nullptr, 0, 0, nullptr, 0, params,
                    out_ids, stream);
}

extern "C" lp_status lp_mask_and_sample(const void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                        int64_t logits_stride, const int32_t* bitmask,
                                        int64_t bitmask_rows, int64_t bitmask_words,
                                        int64_t bitmask_stride, int64_t vocab_size,
                                        const int32_t* indices, int64_t num_indices,
                                        const lp_sampling_params* params, int64_t* out_ids,
                                        cudaStream_t stream) {
  if (!(dt == LP_F32 || dt == LP_F16 || dt == LP_BF16)) return LP_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || cols < 0 || logits_stride < cols || num_indices < 0 ||
      (num_indices > 0 && indices == nullptr))
    return LP_ERR_INVALID_ARGUMENT;
  if (bitmask == nullptr) {
    const int64_t vocab = vocab_size < 0 ? cols : vocab_size;
    if (vocab > cols) return LP_ERR_INVALID_ARGUMENT;
    return run_sample(logits, dt, B, vocab, logits_stride, nullptr, 0, 0, nullptr, 0, params,
                      out_ids, stream);
  }
  if (bitmask_words < 0 || bitmask_stride < bitmask_words || bitmask_rows < 0)
    return LP_ERR_INVALID_ARGUMENT;
  const int64_t capw = bitmask_words * 32;
  const int64_t vocab = vocab_size < 0 ? std::min(cols, capw) : vocab_size;
  if (vocab > cols || vocab > capw) return LP_ERR_INVALID_ARGUMENT;
  if (indices == nullptr && bitmask_rows < B) return LP_ERR_INVALID_ARGUMENT;
  const bool any_masked = indices == nullptr || num_indices > 0;
  return run_sample(logits, dt, B, vocab, logits_stride, any_masked ? bitmask : nullptr,
                    bitmask_rows, bitmask_stride, indices, num_indices, params, out_ids, stream);
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
    case LP_ERR_TOO_LARGE: return "row too long for the sampler";
    default: return "unknown status";
  }
}
