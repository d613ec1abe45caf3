// sample.cu -- fused bitmask + temperature + top-k ∩ top-p ∩ min-p + Gumbel-max
// sampler (Kernel Hub "logits-processor", Ops "sample" and "How it works";
// unsatisfiable rows as in TensorRT-Edge-LLM "Guided Decoder").
//
// GB300 design.  One row is owned by a thread-block cluster of C CTAs (C in
// {1, 2, 4, 8}); each CTA stages its contiguous chunk of the row (and of the
// row's bitmask) in shared memory with cp.async, so HBM is read exactly once and
// every later pass runs on chip.  The CTAs combine partial results through
// distributed shared memory (DSMEM) behind hardware cluster barriers -- no global
// scratch, no atomics on global memory, no spin-waits.
//
// Per row:
//   P1  candidate max / argmax / count (overlapped with the staged loads);
//       cluster reduce.  No candidate -> -1; greedy -> argmax.
//   P2  (top-p only) S = sum of exp((x - max) / T) over candidates.
//   cut a lower bound on the final keep-threshold from whichever filter can
//       certify one: min-p exactly, top-k from the k-th largest per-thread
//       maximum, top-p from the tail-mass bound (candidates below the cut carry
//       at most (1 - top_p) S); candidates at or above it are compacted (P3) into
//       a per-CTA buffer.
//   sel the keep-threshold max(t_k, t_p, t_m) by an MSD radix select over the
//       order-preserving key of the logit (counts for top-k, fixed-point softmax
//       mass for top-p, summed across the cluster per digit).  Top-k and top-p
//       share one descent: the threshold is the largest key at which either
//       "count >= k" or "mass >= top_p * S" first holds.  The descent runs over
//       the compacted buffers; if they overflowed or do not reach the threshold
//       it runs again over the staged chunks (exact in every case).
//   draw Gumbel-max over the kept set with Philox4x32-10 noise keyed by
//       (seed, row, offset); rows without filters draw over all candidates that
//       can still win (z >= z_max - (g_max - g_min)), pruning any token whose best
//       possible score is below the running best.
// Masses are 2^-40 fixed point in 64-bit integers, so every sum is exact and
// order-independent: results are deterministic in (seed, offset).
#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace lp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 4;
constexpr int kKBins = 128;             // log-spaced bins of (max - thread max)
constexpr int kKBase = (127 - 6) << 3;  // code of 2^-6 (8 exponent + 3 fraction bits)
constexpr int kMaxCluster = 8;
constexpr int kDefaultCap = 4096;
constexpr float kLog2e = 1.4426950408889634f;
constexpr double kFix = 1099511627776.0;  // 2^40

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
  int chunk;   // tokens per CTA (multiple of 32)
  int cap;     // compaction buffer entries per CTA
  int mw_off;  // byte offset of the staged bitmask words in dynamic shared memory
  int buf_off; // byte offset of the compaction buffer
};

struct Xchg {  // per-CTA values read by the other CTAs of the cluster
  float max;
  int arg;
  int ncand;
  float sum;
  int count;
  int overflow;
  float best;
  int best_v;
  unsigned kcnt[kKBins];
};

struct Hist {  // double-buffered radix histograms
  unsigned long long mass[2][256];
  unsigned cnt[2][256];
};

__device__ __forceinline__ void arg_combine(float& s, int& v, float s2, int v2) {
  if (s2 > s || (s2 == s && v2 < v)) {
    s = s2;
    v = v2;
  }
}

__device__ __forceinline__ void warp_argmax(float& s, int& v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float s2 = __shfl_xor_sync(kFullWarp, s, o);
    const int v2 = __shfl_xor_sync(kFullWarp, v, o);
    arg_combine(s, v, s2, v2);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFullWarp, x, o);
  return x;
}

__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFullWarp, x, o);
  return x;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    default: cp_async_wait<3>(); break;
  }
}

// Log-spaced bin of d >= 0: bin 0 holds d < 2^-6, bin j >= 1 holds d in
// [2^-6 ... ) with 8 bins per octave; the last bin also holds everything larger.
__device__ __forceinline__ int kbin(float d) {
  const int code = int(__float_as_uint(d) >> 20);
  return min(max(code - kKBase + 1, 0), kKBins - 1);
}
// Exclusive upper edge of bin j (j < kKBins - 1).
__device__ __forceinline__ float kbin_hi(int j) {
  return j == 0 ? 0.015625f : __uint_as_float(unsigned(j + kKBase) << 20);
}

// Per-CTA view of the staged chunk: token v = start + i for local element i.
template <int DT>
struct Chunk {
  using E = Elt<DT>;
  static constexpr int EPV = E::kPerVec;
  static constexpr int EB = E::kBytes;
  const unsigned char* data;  // 16-byte aligned window; element i at byte mis + i*EB
  const uint32_t* mw;         // staged bitmask words of the chunk
  int mis, n_local, nvec, nwords, start;
  bool masked;

  // candidate bits of vector q: element e is a token of this chunk and kept by the mask
  __device__ __forceinline__ uint32_t bits(int q, int& i0) const {
    i0 = (16 * q - mis) / EB;
    const int lo = i0 < 0 ? -i0 : 0;
    const int hi = min(EPV, n_local - i0);
    uint32_t valid = hi > lo ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
    if (!masked || !valid) return valid;
    const int w = i0 >> 5;  // floor division, -1 for a negative i0
    const int sh = i0 & 31;
    const uint32_t w0 = w >= 0 ? mw[w] : 0u;
    const uint32_t w1 = (sh + EPV > 32 && w + 1 < nwords) ? mw[w + 1] : 0u;
    const uint32_t m = uint32_t(((uint64_t(w1) << 32) | w0) >> sh);
    return valid & m;
  }
  __device__ __forceinline__ uint4 vec(int q) const {
    return *reinterpret_cast<const uint4*>(data + 16 * q);
  }
};

template <int DT>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
  using E = Elt<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int EB = E::kBytes;
  constexpr int kLastShift = E::kLowKeyBit & ~7;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int b = int(blockIdx.x) / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* smw = reinterpret_cast<uint32_t*>(smem + a.mw_off);
  float* bval = reinterpret_cast<float*>(smem + a.buf_off);
  int* bidx = reinterpret_cast<int*>(smem + a.buf_off + 4 * a.cap);

  __shared__ Xchg xchg;
  __shared__ Hist hist;
  __shared__ float red_f[kWarps];
  __shared__ int red_i[kWarps];
  __shared__ int red_n[kWarps];
  __shared__ unsigned scan_c[kWarps];
  __shared__ unsigned long long scan_m[kWarps];
  __shared__ unsigned kmerge[kKBins];
  __shared__ int s_count, s_sel;
  __shared__ unsigned s_above_c;
  __shared__ unsigned long long s_above_m;

  // ---------------------------------------------------------------- row setup
  const float T = a.temp ? a.temp[b] : a.temp_s;
  int k = a.topk ? a.topk[b] : a.topk_s;
  const float tp = a.topp ? a.topp[b] : a.topp_s;
  const float mp = a.minp ? a.minp[b] : a.minp_s;

  bool masked = false;
  if (a.bitmask) {
    if (a.indices == nullptr) {
      masked = true;
    } else {
      int found = 0;
      for (int i = tid; i < a.n_indices; i += kThreads) found |= (a.indices[i] == b);
      masked = __syncthreads_or(found) != 0 && b < a.bm_rows;
    }
  }

  Chunk<DT> ch;
  ch.start = rank * a.chunk;
  ch.n_local = max(0, min(a.chunk, a.V - ch.start));
  const char* gsrc = a.logits + int64_t(b) * a.stride_bytes + int64_t(ch.start) * EB;
  ch.mis = int(reinterpret_cast<uintptr_t>(gsrc) & 15);
  const char* g0 = gsrc - ch.mis;
  const int win = ch.mis + ch.n_local * EB;
  ch.nvec = (win + 15) >> 4;
  ch.nwords = (ch.n_local + 31) >> 5;
  ch.data = smem;
  ch.mw = smw;
  ch.masked = masked;

  if (tid < kKBins) xchg.kcnt[tid] = 0u;
  if (tid == 0) s_count = 0;

  // staged loads: full 16-byte vectors by cp.async in kStages groups, the ragged
  // first and last vectors element by element
  const int qf0 = (ch.mis + 15) >> 4;  // first vector wholly inside the window
  const int qf1 = win >> 4;            // vectors [qf0, qf1) are whole
  const int nfull = max(0, qf1 - qf0);
  if (masked) {
    const uint32_t* mrow = a.bitmask + int64_t(b) * a.bm_stride + (ch.start >> 5);
    for (int i = tid; i < ch.nwords; i += kThreads) smw[i] = __ldg(mrow + i);
  }
  if (ch.n_local > 0) {
    if (tid < EPV && ch.mis != 0) {  // ragged first vector
      const int off = tid * EB;
      if (off >= ch.mis && off < win)
        E::store1(reinterpret_cast<char*>(smem) + off, E::bits1(g0 + off));
    }
    if (tid >= 32 && tid < 32 + EPV && (win & 15) != 0 && qf1 >= qf0) {  // ragged last vector
      const int off = 16 * qf1 + (tid - 32) * EB;
      if (off >= ch.mis && off < win)
        E::store1(reinterpret_cast<char*>(smem) + off, E::bits1(g0 + off));
    }
  }
  for (int s = 0; s < kStages; ++s) {
    const int lo = qf0 + int(int64_t(nfull) * s / kStages);
    const int hi = qf0 + int(int64_t(nfull) * (s + 1) / kStages);
    for (int q = lo + tid; q < hi; q += kThreads) cp_async16(smem + 16 * q, g0 + 16 * q);
    cp_async_commit();
  }

  // ------------------------------------------------ P1: max, argmax, count
  float tmax = -INFINITY;
  int targ = INT_MAX;
  int tcnt = 0;
  auto p1_vec = [&](int q) {
    int i0;
    const uint32_t cb = ch.bits(q, i0);
    if (!cb) return;
    const uint4 raw = ch.vec(q);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      if (!((cb >> e) & 1u)) continue;
      const float x = E::get(raw, e);
      if (!(x > -INFINITY)) continue;
      ++tcnt;
      const int v = ch.start + i0 + e;
      if (x > tmax || (x == tmax && v < targ)) {
        tmax = x;
        targ = v;
      }
    }
  };
  for (int s = 0; s < kStages; ++s) {
    cp_async_wait_dyn(kStages - 1 - s);
    __syncthreads();
    const int lo = qf0 + int(int64_t(nfull) * s / kStages);
    const int hi = qf0 + int(int64_t(nfull) * (s + 1) / kStages);
    for (int q = lo + tid; q < hi; q += kThreads) p1_vec(q);
    if (s == 0) {  // the ragged vectors, loaded before the first barrier
      if (tid == 0 && qf0 > 0 && ch.nvec > 0) p1_vec(0);
      if (tid == 1 && qf1 < ch.nvec && qf1 >= qf0) p1_vec(qf1);
    }
  }
  {
    float m = tmax;
    int v = targ;
    warp_argmax(m, v);
    const int n = warp_sum_i(tcnt);
    if (lane == 0) {
      red_f[warp] = m;
      red_i[warp] = v;
      red_n[warp] = n;
    }
    __syncthreads();
    if (tid == 0) {
      float bm = -INFINITY;
      int bv = INT_MAX, nn = 0;
      for (int w = 0; w < kWarps; ++w) {
        arg_combine(bm, bv, red_f[w], red_i[w]);
        nn += red_n[w];
      }
      xchg.max = bm;
      xchg.arg = bv;
      xchg.ncand = nn;
    }
  }
  cluster.sync();  // #1

  float lmax = -INFINITY;
  int larg = INT_MAX;
  int ncand = 0;
  for (int r = 0; r < C; ++r) {
    const Xchg* p = cluster.map_shared_rank(&xchg, r);
    arg_combine(lmax, larg, p->max, p->arg);
    ncand += p->ncand;
  }

  const bool greedy = !(T > 0.f) || k == 1;
  if (ncand == 0 || greedy) {
    if (rank == 0 && tid == 0) a.out[b] = ncand == 0 ? -1 : larg;
    cluster.sync();
    return;
  }

  // ------------------------------------------------------------ row constants
  if (k > 0 && k >= ncand) k = 0;  // keeps every candidate
  const bool has_k = k > 0;
  const bool has_p = tp < 1.f;
  const bool has_m = mp > 0.f;
  const float c2 = kLog2e / T;
  float fm = -INFINITY;  // min-p: keep x >= fm
  if (has_m) {
    const double lm = double(lmax) + double(T) * log(double(mp));
    fm = fminf(__double2float_ru(lm), lmax);
  }

  float best = -INFINITY;
  int bestv = INT_MAX;
  const uint2 key = make_uint2(uint32_t(a.seed), uint32_t(a.seed >> 32));
  auto score_of = [&](float x, int v, uint4& w4, int& wgrp) {
    const int grp = v >> 2;
    if (grp != wgrp) {
      w4 = philox4x32_10(make_uint4(uint32_t(grp), uint32_t(b), uint32_t(a.offset),
                                    uint32_t(a.offset >> 32)),
                         key);
      wgrp = grp;
    }
    const uint32_t word = (v & 3) == 0 ? w4.x : (v & 3) == 1 ? w4.y : (v & 3) == 2 ? w4.z : w4.w;
    return __fdiv_rn(x, T) + gumbel_from_word(word);
  };
  // Gumbel-max over the candidates of the staged chunk with x >= lo
  auto draw_chunk = [&](float lo) {
    uint4 w4 = make_uint4(0, 0, 0, 0);
    int wgrp = -1;
    for (int q = tid; q < ch.nvec; q += kThreads) {
      int i0;
      const uint32_t cb = ch.bits(q, i0);
      if (!cb) continue;
      const uint4 raw = ch.vec(q);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (!((cb >> e) & 1u)) continue;
        const float x = E::get(raw, e);
        if (!(x >= lo) || !(x > -INFINITY)) continue;
        const float z = __fdiv_rn(x, T);
        if (z + kGumbelMax < best) continue;  // cannot beat this thread's best
        const int v = ch.start + i0 + e;
        arg_combine(best, bestv, score_of(x, v, w4, wgrp), v);
      }
    }
  };
  // Gumbel-max over the compacted buffer entries with x >= lo
  auto draw_buffer = [&](float lo, int n) {
    for (int i = tid; i < n; i += kThreads) {
      const float x = bval[i];
      if (!(x >= lo)) continue;
      uint4 w4;
      int wgrp = -1;
      const int v = bidx[i];
      arg_combine(best, bestv, score_of(x, v, w4, wgrp), v);
    }
  };
  // block + cluster argmax of (best, bestv); rank 0 writes the id
  auto finish_draw = [&]() {
    float m = best;
    int v = bestv;
    warp_argmax(m, v);
    if (lane == 0) {
      red_f[warp] = m;
      red_i[warp] = v;
    }
    __syncthreads();
    if (tid == 0) {
      float bm = -INFINITY;
      int bv = INT_MAX;
      for (int w = 0; w < kWarps; ++w) arg_combine(bm, bv, red_f[w], red_i[w]);
      xchg.best = bm;
      xchg.best_v = bv;
    }
    cluster.sync();
    if (rank == 0 && tid == 0) {
      float bm = -INFINITY;
      int bv = INT_MAX;
      for (int r = 0; r < C; ++r) {
        const Xchg* p = cluster.map_shared_rank(&xchg, r);
        arg_combine(bm, bv, p->best, p->best_v);
      }
      a.out[b] = bv == INT_MAX ? -1 : bv;
    }
    cluster.sync();
  };

  if (!has_k && !has_p && !has_m) {  // unfiltered: one Gumbel-max pass
    const double lo = double(lmax) - double(T) * double(kGumbelMax - kGumbelMin);
    draw_chunk(__double2float_rd(lo));
    finish_draw();
    return;
  }

  // ------------------------------------------------------------ P2: softmax sum
  float S = 0.f;
  if (has_p) {
    float ts = 0.f;
    for (int q = tid; q < ch.nvec; q += kThreads) {
      int i0;
      const uint32_t cb = ch.bits(q, i0);
      if (!cb) continue;
      const uint4 raw = ch.vec(q);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (!((cb >> e) & 1u)) continue;
        const float x = E::get(raw, e);
        if (x > -INFINITY) ts += exp2f((x - lmax) * c2);
      }
    }
    ts = warp_sum(ts);
    if (lane == 0) red_f[warp] = ts;
  }
  const bool kbound = has_k && k <= C * kThreads;
  if (kbound && tmax > -INFINITY) atomicAdd(&xchg.kcnt[kbin(lmax - tmax)], 1u);
  __syncthreads();
  if (has_p && tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += red_f[w];
    xchg.sum = t;
  }
  cluster.sync();  // #2
  if (has_p)
    for (int r = 0; r < C; ++r) S += cluster.map_shared_rank(&xchg, r)->sum;
  if (kbound && tid < kKBins) {
    unsigned m = 0;
    for (int r = 0; r < C; ++r) m += cluster.map_shared_rank(&xchg, r)->kcnt[tid];
    kmerge[tid] = m;
  }
  __syncthreads();

  // --------------------------------------------------- cut (certified bound)
  double cut = -INFINITY;
  if (has_m) cut = fmax(cut, double(fm));
  if (kbound) {
    unsigned cum = 0;
    int jk = -1;
    for (int j = 0; j < kKBins - 1; ++j) {
      cum += kmerge[j];
      if (cum >= unsigned(k)) {
        jk = j;
        break;
      }
    }
    if (jk >= 0) cut = fmax(cut, double(lmax) - double(kbin_hi(jk)));
  }
  if (has_p) {
    double D = log(double(ncand) / (fmax(1.0 - double(tp), 1e-30) * double(S)));
    D = fmax(D, 0.0) * 1.0001 + 1e-4;
    cut = fmax(cut, double(lmax) - double(T) * D);
  }
  const float fcut = cut == -INFINITY ? -INFINITY : __double2float_rd(cut);

  // ------------------------------------------ P3: compact candidates >= cut
  {
    const int iters = (ch.nvec + kThreads - 1) / kThreads;
    for (int it = 0; it < iters; ++it) {
      const int q = it * kThreads + tid;
      uint32_t pass = 0;
      int i0 = 0;
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (q < ch.nvec) {
        const uint32_t cb = ch.bits(q, i0);
        if (cb) {
          raw = ch.vec(q);
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            if (!((cb >> e) & 1u)) continue;
            const float x = E::get(raw, e);
            if (x >= fcut && x > -INFINITY) pass |= 1u << e;
          }
        }
      }
      const int n = __popc(pass);
      if (__any_sync(kFullWarp, n != 0)) {
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFullWarp, incl, o);
          if (lane >= o) incl += y;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(&s_count, incl);
        base = __shfl_sync(kFullWarp, base, 31);
        int pos = base + incl - n;
        while (pass) {
          const int e = __ffs(pass) - 1;
          pass &= pass - 1;
          if (pos < a.cap) {
            bval[pos] = E::get(raw, e);
            bidx[pos] = ch.start + i0 + e;
          }
          ++pos;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    xchg.count = min(s_count, a.cap);
    xchg.overflow = s_count > a.cap;
  }
  cluster.sync();  // #3
  int any_overflow = 0;
  for (int r = 0; r < C; ++r) any_overflow |= cluster.map_shared_rank(&xchg, r)->overflow;
  const int nbuf = xchg.count;

  // -------------------------------------- radix select of the keep-threshold
  unsigned long long P = 0ull;  // fixed-point top-p mass target
  if (has_p) {
    const double t = fmax(double(tp), 0.0) * double(S) * kFix;
    P = t >= 1.8e19 ? ~0ull : static_cast<unsigned long long>(t);
  }
  int npass = 0;
  // Finds the largest key x >= key(lo) with count(>= x) >= k (top-k) or
  // mass(>= x) >= P (top-p).  Returns false when no such key exists.
  auto descend = [&](bool from_buffer, float lo, uint32_t& out_key) -> bool {
    const uint32_t klo = fkey(lo), khi = fkey(lmax);
    const uint32_t diff = klo ^ khi;
    const int hb = diff ? 31 - __clz(diff) : int(E::kLowKeyBit);
    int shift = max(hb - 7, 0);
    shift = max(shift & ~7, kLastShift);  // 8-bit digits aligned to the byte grid
    if (hb >= shift + 8) shift += 8;      // keep the highest differing bit inside
    uint32_t prefix = shift + 8 >= 32 ? 0u : (khi >> (shift + 8)) << (shift + 8);
    unsigned above_c = 0;
    unsigned long long above_m = 0;
    for (;;) {
      const int par = npass & 1;
      ++npass;
      hist.cnt[par][tid] = 0u;
      hist.mass[par][tid] = 0ull;
      if (tid == 0) s_sel = -1;
      __syncthreads();
      const uint32_t himask = shift + 8 >= 32 ? 0u : ~0u << (shift + 8);
      auto add = [&](float x) {
        if (!(x >= lo)) return;
        const uint32_t kx = fkey(x);
        if ((kx ^ prefix) & himask) return;
        const int d = int((kx >> shift) & 255u);
        atomicAdd(&hist.cnt[par][d], 1u);
        if (has_p) {
          const float e = exp2f((x - lmax) * c2);
          atomicAdd(&hist.mass[par][d], __float2ull_rn(e * 1099511627776.0f));
        }
      };
      if (from_buffer) {
        for (int i = tid; i < nbuf; i += kThreads) add(bval[i]);
      } else {
        for (int q = tid; q < ch.nvec; q += kThreads) {
          int i0;
          const uint32_t cb = ch.bits(q, i0);
          if (!cb) continue;
          const uint4 raw = ch.vec(q);
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            if ((cb >> e) & 1u) {
              const float x = E::get(raw, e);
              if (x > -INFINITY) add(x);
            }
        }
      }
      __syncthreads();
      cluster.sync();
      // merge bin tid over the cluster, then a descending inclusive scan
      unsigned c = 0;
      unsigned long long m = 0;
      for (int r = 0; r < C; ++r) {
        const Hist* h = cluster.map_shared_rank(&hist, r);
        c += h->cnt[par][tid];
        m += h->mass[par][tid];
      }
      unsigned sc = c;
      unsigned long long sm = m;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {  // suffix sums within the warp
        const unsigned yc = __shfl_down_sync(kFullWarp, sc, o);
        const unsigned long long ym = __shfl_down_sync(kFullWarp, sm, o);
        if (lane + o < 32) {
          sc += yc;
          sm += ym;
        }
      }
      if (lane == 0) {
        scan_c[warp] = sc;
        scan_m[warp] = sm;
      }
      __syncthreads();
      for (int w = warp + 1; w < kWarps; ++w) {
        sc += scan_c[w];
        sm += scan_m[w];
      }
      const unsigned cc = above_c + sc;
      const unsigned long long cm = above_m + sm;
      const bool ok = cc > 0u && ((has_k && cc >= unsigned(k)) || (has_p && cm >= P));
      if (ok) atomicMax(&s_sel, tid);
      __syncthreads();
      const int sel = s_sel;
      if (sel < 0) return false;
      if (tid == sel) {
        s_above_c = cc - c;
        s_above_m = cm - m;
      }
      __syncthreads();
      above_c = s_above_c;
      above_m = s_above_m;
      prefix |= uint32_t(sel) << shift;
      if (shift <= kLastShift) {
        out_key = prefix;
        return true;
      }
      shift -= 8;
    }
  };

  float thr = fm;
  bool from_buffer = !any_overflow;
  if (has_k || has_p) {
    uint32_t kx = 0;
    bool found = false;
    if (from_buffer) {
      found = descend(true, fcut, kx);
      if (!found && !(has_m && fm >= fcut)) from_buffer = false;
    }
    if (!from_buffer) found = descend(false, fm, kx);
    if (found) thr = fmaxf(key_float(kx), fm);
  }

  // ------------------------------------------------------------------- draw
  if (from_buffer)
    draw_buffer(thr, nbuf);
  else
    draw_chunk(thr);
  finish_draw();
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

constexpr int kStaticSmemMargin = 12 * 1024;   // static shared memory of sample_kernel, rounded up
constexpr int kSmemPerBlockMax = 227 * 1024;
constexpr int64_t kChunkTargetBytes = 48 * 1024;
constexpr int64_t kChunkMaxBytes = LP_MAX_SAMPLE_ROW_BYTES / kMaxCluster;

int num_sms() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
  }();
  return n;
}

struct Plan {
  int C, chunk, cap, mw_off, buf_off, smem;
  lp_status status;
};

Plan plan_sample(int64_t B, int64_t V, int eb) {
  Plan p{};
  auto chunk_for = [&](int C) {
    int64_t c = (V + C - 1) / C;
    c = (c + 31) / 32 * 32;
    return std::max<int64_t>(c, 32);
  };
  int C = 1;
  while (C < kMaxCluster && chunk_for(C) * eb > kChunkTargetBytes) C *= 2;
  while (C < kMaxCluster && B * C < 2 * num_sms() && chunk_for(2 * C) >= 4096) C *= 2;
  const int64_t chunk = chunk_for(C);
  if (chunk * eb > kChunkMaxBytes) {
    p.status = LP_ERR_TOO_LARGE;
    return p;
  }
  p.C = C;
  p.chunk = int(chunk);
  const int data = int((chunk * eb + 32 + 15) / 16 * 16);
  const int mw = int((chunk / 32 * 4 + 15) / 16 * 16);
  int cap = kDefaultCap;
  while (cap > 256 && data + mw + 8 * cap + kStaticSmemMargin > kSmemPerBlockMax) cap /= 2;
  p.cap = cap;
  p.mw_off = data;
  p.buf_off = data + mw;
  p.smem = data + mw + 8 * cap;
  p.status = LP_OK;
  return p;
}

template <int DT>
cudaError_t launch_sample(const SampleArgs& a, const Plan& p, int B, cudaStream_t s) {
  static std::mutex mu;
  static int configured = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (p.smem > configured) {
      cudaError_t e = cudaFuncSetAttribute(sample_kernel<DT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
      if (e != cudaSuccess) return e;
      configured = p.smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B) * unsigned(p.C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(p.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(p.C);
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
  if (B > 0x7fffffff / kMaxCluster || vocab > 0x7fffffff || num_indices > 0x7fffffff)
    return LP_ERR_TOO_LARGE;
  const int eb = dt == LP_F32 ? 4 : 2;
  const Plan p = plan_sample(B, vocab, eb);
  if (p.status != LP_OK) return p.status;
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
  a.chunk = p.chunk;
  a.cap = p.cap;
  a.mw_off = p.mw_off;
  a.buf_off = p.buf_off;
  cudaError_t e;
  switch (dt) {
    case LP_F32: e = launch_sample<LP_F32>(a, p, int(B), stream); break;
    case LP_F16: e = launch_sample<LP_F16>(a, p, int(B), stream); break;
    default: e = launch_sample<LP_BF16>(a, p, int(B), stream); break;
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
