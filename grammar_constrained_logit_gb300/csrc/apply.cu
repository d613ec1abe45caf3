// apply.cu -- packed-bitmask apply (XGrammar "Bitmask Operations",
// apply_token_bitmask_inplace; Modular MAX "apply_packed_bitmask").
//
// One streaming pass over the selected rows.  Each thread owns whole 16-byte
// vectors of a row (4 float32 or 8 half/bfloat16 tokens) and reads the one or two
// bitmask words that cover them (consecutive lanes share a word, so the warp's
// mask read is one broadcast-coalesced sector).  In place nothing is read but
// the bitmask: a vector whose tokens are all kept is not touched, a vector whose
// tokens are all masked is written with the fill pattern, and in a mixed vector
// only the masked elements are written (element or element-pair stores).  Out of
// place, every vector of every row is written once (masked rows blended, other
// rows copied).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"

namespace lp {
namespace {

constexpr int kApplyThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int kVecPerBlock = kApplyThreads * kVecPerThread;
constexpr int kReportBatch = 4;  // mask words a thread loads at once for the report

struct ApplyArgs {
  char* out;                  // out of place: destination rows
  int64_t out_stride;         // bytes
  const char* in;             // logits rows (also the destination in place)
  int64_t in_stride;          // bytes
  int64_t B, cols, vocab;
  const uint32_t* bitmask;    // [bitmask_rows, bm_stride] words
  int64_t bm_stride, bm_rows;
  const int32_t* indices;     // selected rows, or nullptr
  int64_t n_indices;
  const uint8_t* row_flags;   // in place, no indices: row b masked iff row_flags[b] != 0
  int32_t* has_token;         // in place: has_token[b] = 1 when row b keeps a token, else 0
  int64_t n_rows;             // row slots walked by blockIdx.y
  uint32_t fill;              // fill bit pattern of one element
  int use_bitmap;             // out of place with indices: selection bitmap in shared memory
  int copy_only;              // out of place: treat every row as unselected
  int vec_ok;                 // out of place: source and destination rows share the 16-byte phase
};

__device__ __forceinline__ uint4 ld_stream(const char* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
// Stores keep the default L2 priority: the masked logits are what the sampler
// reads next, and evict-first lines would be written back while the next
// launch's bitmask reads wait on the memory.
__device__ __forceinline__ void st_vec(char* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// The fill pattern into the masked elements of one 16-byte vector (bit e of keep
// set: element e kept and left alone).
template <int DT>
__device__ __forceinline__ void store_masked(char* p, uint32_t keep, uint32_t fill_w) {
  if constexpr (DT == LP_F32) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (!((keep >> e) & 1u)) *(reinterpret_cast<unsigned*>(p) + e) = fill_w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // element pair i is 32-bit word i
      const uint32_t m = (~keep >> (2 * i)) & 3u;
      if (m == 3u)
        *(reinterpret_cast<unsigned*>(p) + i) = fill_w;
      else if (m == 1u)
        *(reinterpret_cast<unsigned short*>(p) + 2 * i) = static_cast<unsigned short>(fill_w);
      else if (m == 2u)
        *(reinterpret_cast<unsigned short*>(p) + 2 * i + 1) =
            static_cast<unsigned short>(fill_w >> 16);
    }
  }
}

template <int DT, bool OOP>
__global__ void __launch_bounds__(kApplyThreads) apply_kernel(const ApplyArgs a) {
  using E = Elt<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int EB = E::kBytes;
  constexpr uint32_t ALL = (1u << EPV) - 1u;
  constexpr int64_t kChunkElems = int64_t(kVecPerBlock) * EPV;
  extern __shared__ uint32_t sel_bitmap[];

  const int64_t sel_limit = a.B < a.bm_rows ? a.B : a.bm_rows;
  if (OOP && a.use_bitmap) {
    const int nw = int((a.B + 31) >> 5);
    for (int i = threadIdx.x; i < nw; i += blockDim.x) sel_bitmap[i] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < a.n_indices; i += blockDim.x) {
      const int64_t r = a.indices[i];
      if (r >= 0 && r < sel_limit) atomicOr(&sel_bitmap[r >> 5], 1u << (r & 31));
    }
    __syncthreads();
  }
  const uint32_t fill_w = E::fill_word(a.fill);
  const uint4 fill_v = make_uint4(fill_w, fill_w, fill_w, fill_w);

  for (int64_t slot = blockIdx.y; slot < a.n_rows; slot += gridDim.y) {
    int64_t b;
    bool sel;
    if (OOP) {
      b = slot;
      if (a.copy_only)
        sel = false;
      else if (a.use_bitmap)
        sel = (sel_bitmap[b >> 5] >> (b & 31)) & 1u;
      else
        sel = true;
    } else {
      b = a.indices ? int64_t(a.indices[slot]) : slot;
      if (b < 0 || b >= sel_limit) continue;  // invalid index: skipped
      sel = a.row_flags == nullptr || a.row_flags[b] != 0;
    }
    const char* rin = a.in + b * a.in_stride;
    char* rout = OOP ? a.out + b * a.out_stride : const_cast<char*>(rin);
    const uint32_t* mrow = a.bitmask + b * a.bm_stride;
    const int64_t limit = sel ? a.vocab : 0;  // tokens >= limit are kept
    const int64_t n_el = OOP ? a.cols : a.vocab;

    int64_t head, nvec;
    if (!OOP || a.vec_ok) {
      const int mis = int(reinterpret_cast<uintptr_t>(rin) & 15);
      head = ((16 - mis) & 15) / EB;
      if (head > n_el) head = n_el;
      nvec = (n_el - head) / EPV;
    } else {
      head = n_el;  // rows out of phase: element by element
      nvec = 0;
    }
    const int64_t tail0 = head + nvec * EPV;

    // scalar elements (ragged head and tail, or whole rows out of phase) of this
    // block's element range
    const int64_t e_lo = int64_t(blockIdx.x) * kChunkElems;
    const int64_t e_hi = e_lo + kChunkElems;
    auto scalar = [&](int64_t j) {
      const bool keep = sel ? (mask_bits(mrow, j, 1, limit) & 1u) : true;
      if (OOP)
        E::store1(rout + j * EB, keep ? E::bits1(rin + j * EB) : a.fill);
      else if (!keep)
        E::store1(rout + j * EB, a.fill);
    };
    for (int64_t j = e_lo + threadIdx.x; j < e_hi && j < head; j += blockDim.x) scalar(j);
    for (int64_t j = (e_lo > tail0 ? e_lo : tail0) + threadIdx.x; j < e_hi && j < n_el;
         j += blockDim.x)
      scalar(j);

    // whole vectors of this block's vector range: every mask word, then (out of
    // place) every logits vector that must be read, then the stores, so that one
    // thread's loads are all in flight together (a store may alias a later load,
    // which would otherwise hold that load back behind it)
    int64_t j0[kVecPerThread];
    uint32_t keep[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t q = int64_t(blockIdx.x) * kVecPerBlock + k * kApplyThreads + threadIdx.x;
      j0[k] = head + q * EPV;
      // with row flags the mask words load beside the flag, not after it
      keep[k] = q >= nvec                        ? ~0u
                : sel || a.row_flags != nullptr ? mask_bits(mrow, j0[k], EPV, a.vocab)
                                                 : ALL;
    }
    if (!sel) {
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) keep[k] = keep[k] == ~0u ? ~0u : ALL;
    }
    uint4 v[kVecPerThread];
    if (OOP) {
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k)
        if (keep[k] != ~0u && keep[k] != 0u) v[k] = ld_stream(rin + j0[k] * EB);
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      if (keep[k] == ~0u || (!OOP && keep[k] == ALL)) continue;
      char* const dst = rout + j0[k] * EB;
      if (!OOP && keep[k] != 0u) {
        store_masked<DT>(dst, keep[k], fill_w);
        continue;
      }
      const uint4 w = keep[k] == 0u ? fill_v : keep[k] == ALL ? v[k] : E::blend(v[k], keep[k], a.fill);
      st_vec(dst, w);
    }
    // block-uniform: the row's first block reports the whole row (its words below
    // vocab_size; an unflagged row keeps every token).  The mask bits of its own
    // vectors, already loaded, settle most flagged rows; the others read every
    // word of the row, kReportBatch independent loads a thread at a time.
    if (!OOP && a.has_token != nullptr && blockIdx.x == 0) {
      bool kept = !sel && a.vocab > 0;
      if (sel) {
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) kept |= keep[k] != ~0u && keep[k] != 0u;
      }
      if (sel && !__syncthreads_or(kept)) {
        const int64_t nw = (a.vocab + 31) >> 5;
        const uint32_t last = (a.vocab & 31) ? (1u << (a.vocab & 31)) - 1u : ~0u;
        for (int64_t w0 = threadIdx.x; w0 < nw; w0 += int64_t(kReportBatch) * blockDim.x) {
          uint32_t wd[kReportBatch];
#pragma unroll
          for (int u = 0; u < kReportBatch; ++u) {
            const int64_t w = w0 + int64_t(u) * blockDim.x;
            wd[u] = w < nw ? __ldg(mrow + w) & (w == nw - 1 ? last : ~0u) : 0u;
          }
#pragma unroll
          for (int u = 0; u < kReportBatch; ++u) kept |= wd[u] != 0u;
        }
      }
      const int r = __syncthreads_or(kept);
      if (threadIdx.x == 0) a.has_token[b] = r ? 1 : 0;
    }
  }
}

// ------------------------------------------------------------------- host

int elt_bytes(lp_dtype dt) { return dt == LP_F32 ? 4 : 2; }

bool dtype_ok(lp_dtype dt) { return dt == LP_F32 || dt == LP_F16 || dt == LP_BF16; }

template <bool OOP>
cudaError_t launch_apply(lp_dtype dt, const ApplyArgs& a, int64_t max_elems, cudaStream_t s) {
  const int EPV = dt == LP_F32 ? 4 : 8;
  const int64_t chunk = int64_t(kVecPerBlock) * EPV;
  const int64_t gx = (max_elems + chunk - 1) / chunk + 1;
  const int64_t gy = std::min<int64_t>(a.n_rows, 65535);
  if (gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const dim3 grid{static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u};
  const size_t smem = (OOP && a.use_bitmap) ? size_t((a.B + 31) / 32) * 4 : 0;
  switch (dt) {
    case LP_F32:
      if (smem > 48 * 1024)
        cudaFuncSetAttribute(apply_kernel<LP_F32, OOP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      apply_kernel<LP_F32, OOP><<<grid, kApplyThreads, smem, s>>>(a);
      break;
    case LP_F16:
      if (smem > 48 * 1024)
        cudaFuncSetAttribute(apply_kernel<LP_F16, OOP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      apply_kernel<LP_F16, OOP><<<grid, kApplyThreads, smem, s>>>(a);
      break;
    default:
      if (smem > 48 * 1024)
        cudaFuncSetAttribute(apply_kernel<LP_BF16, OOP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      apply_kernel<LP_BF16, OOP><<<grid, kApplyThreads, smem, s>>>(a);
      break;
  }
  return cudaGetLastError();
}

// Round-to-nearest-even of a float into the element type's bit pattern, by
// CUDA's own host-side conversions.
uint32_t fill_bits(float f, lp_dtype dt) {
  if (dt == LP_F32) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
  }
  if (dt == LP_F16) {
    const __half_raw r = __float2half_rn(f);
    return r.x;
  }
  const __nv_bfloat16_raw r = __float2bfloat16_rn(f);
  return r.x;
}

struct Geometry {
  int64_t vocab;
  lp_status status;
};

Geometry check_common(lp_dtype dt, int64_t B, int64_t cols, int64_t logits_stride,
                      int64_t bitmask_rows, int64_t bitmask_words, int64_t bitmask_stride,
                      int64_t vocab_size, const int32_t* indices, int64_t num_indices) {
  Geometry g{0, LP_OK};
  if (!dtype_ok(dt)) {
    g.status = LP_ERR_UNSUPPORTED_DTYPE;
    return g;
  }
  if (B < 0 || cols < 0 || logits_stride < cols || bitmask_words < 0 ||
      bitmask_stride < bitmask_words || bitmask_rows < 0 || num_indices < 0 ||
      (num_indices > 0 && indices == nullptr)) {
    g.status = LP_ERR_INVALID_ARGUMENT;
    return g;
  }
  const int64_t cap = bitmask_words * 32;
  g.vocab = vocab_size < 0 ? std::min(cols, cap) : vocab_size;
  if (g.vocab > cols || g.vocab > cap) g.status = LP_ERR_INVALID_ARGUMENT;
  if (indices == nullptr && bitmask_rows < B) g.status = LP_ERR_INVALID_ARGUMENT;
  return g;
}

}  // namespace
}  // namespace lp

using namespace lp;

extern "C" lp_status lp_apply_token_bitmask(void* logits, lp_dtype dt, int64_t B, int64_t cols,
                                            int64_t logits_stride, const int32_t* bitmask,
                                            int64_t bitmask_rows, int64_t bitmask_words,
                                            int64_t bitmask_stride, int64_t vocab_size,
                                            const int32_t* indices, int64_t num_indices,
                                            cudaStream_t stream) {
  Geometry g = check_common(dt, B, cols, logits_stride, bitmask_rows, bitmask_words,
                            bitmask_stride, vocab_size, indices, num_indices);
  if (g.status != LP_OK) return g.status;
  const int64_t rows = indices ? num_indices : B;
  if (B == 0 || g.vocab == 0 || rows == 0) return LP_OK;
  if (logits == nullptr || bitmask == nullptr) return LP_ERR_INVALID_ARGUMENT;
  const int64_t eb = elt_bytes(dt);
  ApplyArgs a{};
  a.out = static_cast<char*>(logits);
  a.out_stride = logits_stride * eb;
  a.in = static_cast<const char*>(logits);
  a.in_stride = logits_stride * eb;
  a.B = B;
  a.cols = cols;
  a.vocab = g.vocab;
  a.bitmask = reinterpret_cast<const uint32_t*>(bitmask);
  a.bm_stride = bitmask_stride;
  a.bm_rows = bitmask_rows;
  a.indices = indices;
  a.n_indices = num_indices;
  a.n_rows = rows;
  a.fill = fill_bits(-__builtin_huge_valf(), dt);
  a.vec_ok = 1;
  return launch_apply<false>(dt, a, g.vocab, stream) == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

extern "C" lp_status lp_apply_token_bitmask_rows(void* logits, lp_dtype dt, int64_t B,
                                                 int64_t cols, int64_t logits_stride,
                                                 const int32_t* bitmask, int64_t bitmask_rows,
                                                 int64_t bitmask_words, int64_t bitmask_stride,
                                                 int64_t vocab_size,
                                                 const uint8_t* row_needs_mask,
                                                 int32_t* row_has_token, cudaStream_t stream) {
  Geometry g = check_common(dt, B, cols, logits_stride, bitmask_rows, bitmask_words,
                            bitmask_stride, vocab_size, nullptr, 0);
  if (g.status != LP_OK) return g.status;
  if (B == 0) return LP_OK;
  if (g.vocab > 0 && (logits == nullptr || bitmask == nullptr)) return LP_ERR_INVALID_ARGUMENT;
  if (g.vocab == 0) {  // no row keeps a token, and there is nothing to mask
    if (row_has_token != nullptr &&
        cudaMemsetAsync(row_has_token, 0, size_t(B) * sizeof(int32_t), stream) != cudaSuccess)
      return LP_ERR_CUDA;
    return LP_OK;
  }
  const int64_t eb = elt_bytes(dt);
  ApplyArgs a{};
  a.out = static_cast<char*>(logits);
  a.out_stride = logits_stride * eb;
  a.in = static_cast<const char*>(logits);
  a.in_stride = logits_stride * eb;
  a.B = B;
  a.cols = cols;
  a.vocab = g.vocab;
  a.bitmask = reinterpret_cast<const uint32_t*>(bitmask);
  a.bm_stride = bitmask_stride;
  a.bm_rows = bitmask_rows;
  a.n_rows = B;
  a.row_flags = row_needs_mask;
  a.has_token = row_has_token;
  a.fill = fill_bits(-__builtin_huge_valf(), dt);
  a.vec_ok = 1;
  return launch_apply<false>(dt, a, g.vocab, stream) == cudaSuccess ? LP_OK : LP_ERR_CUDA;
}

extern "C" lp_status lp_apply_packed_bitmask(void* out, int64_t out_stride, const void* logits,
                                             lp_dtype dt, int64_t B, int64_t cols,
                                             int64_t logits_stride, const int32_t* bitmask,
                                             int64_t bitmask_rows, int64_t bitmask_words,
                                             int64_t bitmask_stride, float fill_value,
                                             int64_t vocab_size, const int32_t* indices,
                                             int64_t num_indices, cudaStream_t stream) {
  Geometry g = check_common(dt, B, cols, logits_stride, bitmask_rows, bitmask_words,
                            bitmask_stride, vocab_size, indices, num_indices);
  if (g.status != LP_OK) return g.status;
  if (out_stride < cols) return LP_ERR_INVALID_ARGUMENT;
  if (B == 0 || cols == 0) return LP_OK;
  if (out == nullptr || logits == nullptr) return LP_ERR_INVALID_ARGUMENT;
  const bool any_masking = g.vocab > 0 && (indices == nullptr || num_indices > 0);
  if (any_masking && bitmask == nullptr) return LP_ERR_INVALID_ARGUMENT;
  const int64_t eb = elt_bytes(dt);
  const uint32_t fill = fill_bits(fill_value, dt);

  if (out == logits && out_stride == logits_stride) {  // in place with a fill value
    if (!any_masking) return LP_OK;
    ApplyArgs a{};
    a.out = static_cast<char*>(out);
    a.out_stride = out_stride * eb;
    a.in = static_cast<const char*>(logits);
    a.in_stride = logits_stride * eb;
    a.B = B;
    a.cols = cols;
    a.vocab = g.vocab;
    a.bitmask = reinterpret_cast<const uint32_t*>(bitmask);
    a.bm_stride = bitmask_stride;
    a.bm_rows = bitmask_rows;
    a.indices = indices;
    a.n_indices = num_indices;
    a.n_rows = indices ? num_indices : B;
    a.fill = fill;
    a.vec_ok = 1;
    return launch_apply<false>(dt, a, g.vocab, stream) == cudaSuccess ? LP_OK : LP_ERR_CUDA;
  }

  ApplyArgs a{};
  a.out = static_cast<char*>(out);
  a.out_stride = out_stride * eb;
  a.in = static_cast<const char*>(logits);
  a.in_stride = logits_stride * eb;
  a.B = B;
  a.cols = cols;
  a.vocab = g.vocab;
  a.bitmask = reinterpret_cast<const uint32_t*>(bitmask);
  a.bm_stride = bitmask_stride;
  a.bm_rows = bitmask_rows;
  a.indices = indices;
  a.n_indices = num_indices;
  a.n_rows = B;
  a.fill = fill;
  const uintptr_t po = reinterpret_cast<uintptr_t>(out), pi = reinterpret_cast<uintptr_t>(logits);
  a.vec_ok = ((po - pi) & 15) == 0 && (((out_stride - logits_stride) * eb) & 15) == 0;
  // Rows selected through indices are marked in a per-block bitmap of B bits;
  // past 48 KB of bitmap, copy every row first and mask the selected rows in place.
  const bool big_bitmap = indices != nullptr && (B + 31) / 32 * 4 > 48 * 1024;
  if (!any_masking || big_bitmap) a.copy_only = 1;
  else if (indices != nullptr) a.use_bitmap = 1;
  if (launch_apply<true>(dt, a, cols, stream) != cudaSuccess) return LP_ERR_CUDA;
  if (big_bitmap && any_masking) {
    ApplyArgs m = a;
    m.out = static_cast<char*>(out);
    m.out_stride = out_stride * eb;
    m.in = static_cast<const char*>(out);
    m.in_stride = out_stride * eb;
    m.use_bitmap = 0;
    m.copy_only = 0;
    m.vec_ok = 1;
    m.n_rows = num_indices;
    if (launch_apply<false>(dt, m, g.vocab, stream) != cudaSuccess) return LP_ERR_CUDA;
  }
  return LP_OK;
}
