// vocab_argmax_topk: per-row argmax, top-k (value desc, index asc), max and
// log-sum-exp of next-token logits (Graft page §2 second/third gears: table
// rows hold the top-k successors, refreshed from every verified position;
// greedy verification compares with the target's argmax).
//
// HBM-bound streaming design:
//   pass 1  grid (chunks, rows): a CTA of 256 threads owns an 8192-element
//           chunk of one row, held in registers (32 values per thread, loaded
//           with 16-byte streaming loads).  It computes the chunk max, the sum
//           of exp(x - max) and the chunk's top-k.  For the top-k it first
//           takes tau = k-th largest of the 256 per-thread maxima: at least k
//           elements are >= tau, so every member of the chunk top-k is too.
//           Only elements >= tau (typically a dozen) are ranked.
//   pass 2  one warp per row merges the chunk partials in chunk order
//           (deterministic) and writes the outputs.
#include <cuda_bf16.h>
#include <float.h>

#include <algorithm>
#include <cstdlib>

#include "tv_common.cuh"

namespace tv {

constexpr int kVThreads = 256;
constexpr int kVPerThread = 32;
constexpr int kVChunk = kVThreads * kVPerThread;   // 8192 elements
constexpr int kVCandCap = 1024;

template <int KMAX>
struct VocabPart {
  float m, s;
  float val[KMAX];
  int idx[KMAX];
};

// 8 consecutive elements starting at e0 (e0 multiple of 8).  Out-of-range
// entries become -inf.  `vec_ok` says whether 16-byte vector loads are legal.
__device__ __forceinline__ void load8(const uint16_t* row, int e0, int V, bool vec_ok, float* o) {
  if (vec_ok && e0 + 8 <= V) {
    uint4 w = ldg_stream(row + e0);
    o[0] = bf16_lo(w.x); o[1] = bf16_hi(w.x); o[2] = bf16_lo(w.y); o[3] = bf16_hi(w.y);
    o[4] = bf16_lo(w.z); o[5] = bf16_hi(w.z); o[6] = bf16_lo(w.w); o[7] = bf16_hi(w.w);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = (e0 + q < V) ? bf16_at(row + e0 + q) : -INFINITY;
  }
}

__device__ __forceinline__ void load8(const float* row, int e0, int V, bool vec_ok, float* o) {
  if (vec_ok && e0 + 8 <= V) {
    uint4 a = ldg_stream(row + e0);
    uint4 b = ldg_stream(row + e0 + 4);
    o[0] = __uint_as_float(a.x); o[1] = __uint_as_float(a.y);
    o[2] = __uint_as_float(a.z); o[3] = __uint_as_float(a.w);
    o[4] = __uint_as_float(b.x); o[5] = __uint_as_float(b.y);
    o[6] = __uint_as_float(b.z); o[7] = __uint_as_float(b.w);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = (e0 + q < V) ? row[e0 + q] : -INFINITY;
  }
}

// Insert (v, i) into the sorted list (tv, ti) of length K if it belongs there.
template <int K>
__device__ __forceinline__ void list_insert(float* tv, int* ti, float v, int i) {
  if (!better(v, i, tv[K - 1], ti[K - 1])) return;
  tv[K - 1] = v;
  ti[K - 1] = i;
#pragma unroll
  for (int q = K - 1; q > 0; --q) {
    if (better(tv[q], ti[q], tv[q - 1], ti[q - 1])) {
      float a = tv[q]; tv[q] = tv[q - 1]; tv[q - 1] = a;
      int b = ti[q]; ti[q] = ti[q - 1]; ti[q - 1] = b;
    }
  }
}

// K rounds of warp-wide "pop the best head" over per-lane sorted lists.
// Every lane ends with the merged list in (ov, oi).
template <int K>
__device__ __forceinline__ void warp_merge_lists(float* tv, int* ti, float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < K; ++t) {
    float bv = tv[0];
    int bi = ti[0];
    int bl = lane;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      int l2 = __shfl_xor_sync(0xffffffffu, bl, o);
      if (better(v2, i2, bv, bi) || (v2 == bv && i2 == bi && l2 < bl)) {
        bv = v2; bi = i2; bl = l2;
      }
    }
    ov[t] = bv;
    oi[t] = bi;
    if (lane == bl) {
#pragma unroll
      for (int q = 0; q < K - 1; ++q) { tv[q] = tv[q + 1]; ti[q] = ti[q + 1]; }
      tv[K - 1] = -INFINITY;
      ti[K - 1] = INT32_MAX;
    }
  }
}

template <typename T, int KMAX, bool LSE>
__global__ void __launch_bounds__(kVThreads) vocab_partial_kernel(
    const T* __restrict__ logits, int V, int64_t ld, const int32_t* __restrict__ row_idx,
    bool vec_ok, VocabPart<KMAX>* __restrict__ part) {
  __shared__ float s_red[kVThreads / 32];
  __shared__ float s_wtop[kVThreads / 32][KMAX];
  __shared__ int s_wcnt[kVThreads / 32];
  __shared__ float s_cv[kVCandCap];
  __shared__ int s_ci[kVCandCap];
  __shared__ float s_bc[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x;
  const int row = blockIdx.y;
  const int src = row_idx ? row_idx[row] : row;
  const T* x = logits + static_cast<int64_t>(src) * ld;
  const int base = chunk * kVChunk;

  float v[kVPerThread];
#pragma unroll
  for (int j = 0; j < kVPerThread / 8; ++j)
    load8(x, base + (j * kVThreads + tid) * 8, V, vec_ok, v + 8 * j);
  auto eidx = [&](int t) { return base + ((t >> 3) * kVThreads + tid) * 8 + (t & 7); };

  // ---- chunk max
  float m = v[0];
#pragma unroll
  for (int t = 1; t < kVPerThread; ++t) m = fmaxf(m, v[t]);
  const float my_max = m;
  m = warp_max(m);
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float mm = s_red[0];
#pragma unroll
    for (int w = 1; w < kVThreads / 32; ++w) mm = fmaxf(mm, s_red[w]);
    s_bc[0] = mm;
  }

  // ---- tau = KMAX-th largest per-thread maximum (values only)
  {
    float mv = my_max;
    for (int t = 0; t < KMAX; ++t) {
      float b = warp_max(mv);
      unsigned hit = __ballot_sync(0xffffffffu, mv == b);
      if (lane == __ffs(hit) - 1) mv = -INFINITY;
      if (lane == 0) s_wtop[warp][t] = b;
    }
  }
  __syncthreads();
  const float M = s_bc[0];
  if (warp == 0) {
    // merge the 8 per-warp descending lists: lane l < 8 walks list l
    float head = -INFINITY;
    int pos = 0;
    if (lane < kVThreads / 32) head = s_wtop[lane][0];
    float tau = -INFINITY;
    for (int t = 0; t < KMAX; ++t) {
      float b = warp_max(head);
      unsigned hit = __ballot_sync(0xffffffffu, head == b && lane < kVThreads / 32);
      if (lane == __ffs(hit) - 1) {
        ++pos;
        head = pos < KMAX ? s_wtop[lane][pos] : -INFINITY;
      }
      tau = b;
    }
    if (lane == 0) s_bc[1] = tau;
  }

  // ---- sum of exp(x - M) in fp32 (2^((x - M) log2 e) on the SFU)
  float sum = 0.f;
  if (LSE) {
    const float mb = M * kLog2e;
#pragma unroll
    for (int t = 0; t < kVPerThread; ++t) sum += ex2(fmaf(v[t], kLog2e, -mb));
    sum = warp_sum(sum);
  }
  __syncthreads();   // s_bc[1] ready; s_red free for the sums
  if (LSE && lane == 0) s_red[warp] = sum;
  const float tau = s_bc[1];

  // ---- candidates >= tau, compacted in (thread, element) order
  int c = 0;
#pragma unroll
  for (int t = 0; t < kVPerThread; ++t) c += v[t] >= tau;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wcnt[warp] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kVThreads / 32; ++w) {
    const int cw = s_wcnt[w];
    wbase += (w < warp) ? cw : 0;
    total += cw;
  }
  if (total <= kVCandCap) {
    int o = wbase + incl - c;
#pragma unroll
    for (int t = 0; t < kVPerThread; ++t) {
      if (v[t] >= tau) {
        s_cv[o] = v[t];
        s_ci[o] = eidx(t);
        ++o;
      }
    }
  }
  __syncthreads();

  float lv[KMAX];
  int li[KMAX];
#pragma unroll
  for (int q = 0; q < KMAX; ++q) { lv[q] = -INFINITY; li[q] = INT32_MAX; }
  if (total <= kVCandCap) {
    if (warp == 0) {
      for (int t = lane; t < total; t += 32) list_insert<KMAX>(lv, li, s_cv[t], s_ci[t]);
    }
  } else {
    // Pathological ties: every thread ranks its own values, then all warps merge.
#pragma unroll
    for (int t = 0; t < kVPerThread; ++t) list_insert<KMAX>(lv, li, v[t], eidx(t));
  }
  float ov[KMAX];
  int oi[KMAX];
  VocabPart<KMAX>* out = part + static_cast<int64_t>(row) * gridDim.x + chunk;
  if (total <= kVCandCap) {
    if (warp == 0) {
      warp_merge_lists<KMAX>(lv, li, ov, oi);
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < KMAX; ++q) { out->val[q] = ov[q]; out->idx[q] = oi[q]; }
      }
    }
  } else {
    warp_merge_lists<KMAX>(lv, li, ov, oi);
    __syncthreads();   // candidate buffer reused for the per-warp lists
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < KMAX; ++q) { s_cv[warp * KMAX + q] = ov[q]; s_ci[warp * KMAX + q] = oi[q]; }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int q = 0; q < KMAX; ++q) {
        const bool have = lane < kVThreads / 32;
        lv[q] = have ? s_cv[lane * KMAX + q] : -INFINITY;
        li[q] = have ? s_ci[lane * KMAX + q] : INT32_MAX;
      }
      warp_merge_lists<KMAX>(lv, li, ov, oi);
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < KMAX; ++q) { out->val[q] = ov[q]; out->idx[q] = oi[q]; }
      }
    }
  }
  if (tid == 0) {
    out->m = M;
    float s = 0.f;
    if (LSE) {
#pragma unroll
      for (int w = 0; w < kVThreads / 32; ++w) s += s_red[w];
    }
    out->s = s;
  }
}

template <int KMAX, bool LSE>
__global__ void __launch_bounds__(128) vocab_merge_kernel(
    const VocabPart<KMAX>* __restrict__ part, int n_chunks, int rows,
    const int32_t* __restrict__ row_idx, int k, int32_t* __restrict__ argmax,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_val, float* __restrict__ row_max,
    float* __restrict__ row_lse) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int dst = row_idx ? row_idx[row] : row;
  const VocabPart<KMAX>* p = part + static_cast<int64_t>(row) * n_chunks;

  float M = -INFINITY;
  for (int c = lane; c < n_chunks; c += 32) M = fmaxf(M, p[c].m);
  M = warp_max(M);
  float S = 0.f;
  if (LSE) {
    for (int c = lane; c < n_chunks; c += 32) S += p[c].s * ex2((p[c].m - M) * kLog2e);
    S = warp_sum(S);
  }
  float lv[KMAX];
  int li[KMAX];
#pragma unroll
  for (int q = 0; q < KMAX; ++q) { lv[q] = -INFINITY; li[q] = INT32_MAX; }
  for (int c = lane; c < n_chunks; c += 32) {
#pragma unroll
    for (int q = 0; q < KMAX; ++q) list_insert<KMAX>(lv, li, p[c].val[q], p[c].idx[q]);
  }
  float ov[KMAX];
  int oi[KMAX];
  warp_merge_lists<KMAX>(lv, li, ov, oi);
  if (lane == 0) {
    argmax[dst] = oi[0];
    if (row_max) row_max[dst] = M;
    if (LSE && row_lse) row_lse[dst] = M + logf(S);
  }
  if (k > 0 && lane < k) {
    float val = ov[0];
    int idx = oi[0];
#pragma unroll
    for (int q = 1; q < KMAX; ++q)
      if (lane == q) { val = ov[q]; idx = oi[q]; }
    if (topk_idx) topk_idx[static_cast<int64_t>(dst) * k + lane] = idx;
    if (topk_val) topk_val[static_cast<int64_t>(dst) * k + lane] = val;
  }
}

// ---------------------------------------------------------------------------
// Streaming variant (used whenever rows and chunk tails are 16-byte aligned).
//
// A persistent grid of CTAs walks the (row, chunk) items in claim order.  In
// each CTA a producer warp claims items from a global counter (SMs that run
// slower simply take fewer) and copies each 8192-element chunk into the next
// slot of a shared-memory ring with a 1-D bulk copy, a ring's length ahead.
// Compute warp w owns segment w of every chunk: its 1024 contiguous
// elements.  Per segment it records only the maximum and, for the
// log-sum-exp, the sum of exp(x - maximum); there is no block barrier and no
// candidate list, so the warps never wait for one another.
//
// A merge kernel (one warp per row) follows.  Row max = the largest segment
// maximum; log-sum-exp from the segment sums in (chunk, segment) order; the
// top-k threshold tau = the k-th largest segment maximum: k distinct
// elements (one per segment) are >= tau, so every member of the row's top-k
// is >= tau and lies in a segment whose maximum reaches tau (about k of
// them).  Only those segments are read again; their elements >= tau,
// typically a dozen, are ranked exactly by (value desc, index asc).
// ---------------------------------------------------------------------------
// ring of 8192-element chunks: 3 x 16 KB for bf16 (four CTAs per SM), 3 x 32 KB for fp32
template <typename T> constexpr int stream_stages() { return 3; }
template <typename T> constexpr int stream_chunk_bytes() { return kVChunk * static_cast<int>(sizeof(T)); }
constexpr int kSegs = kVThreads / 32;        // segments per chunk = compute warps
constexpr int kSegLen = kVChunk / kSegs;     // 1024 elements
constexpr int kMaxFastSegs = 256;            // segment maxima a merge keeps in registers (8 per lane)

__device__ __forceinline__ uint32_t sm_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (about 2 s); false when it ran out.
__device__ __noinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  if (bar_try(bar, parity)) return true;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (bar_try(bar, parity)) return true;
    if ((i & 63) == 0) {
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 2000000000ull) return false;
    }
  }
  return false;
}
__device__ __forceinline__ bool bar_wait_fast(uint32_t bar, uint32_t parity) {
  return bar_try(bar, parity) || bar_wait(bar, parity);
}
__device__ __forceinline__ void bar_arrive_plain(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Warp-wide float maximum in one instruction (sm_100 family).
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Sort one (value, index) pair per lane by (value desc, index asc): lane 0 best.
__device__ __forceinline__ void warp_bitonic_desc(float& v, int& i) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
      const int oi = __shfl_xor_sync(0xffffffffu, i, stride);
      const bool lower = (lane & stride) == 0;
      const bool desc = (lane & size) == 0;   // this segment ends best-first
      const bool ob = better(ov, oi, v, i);
      if ((lower == desc) ? ob : !ob) { v = ov; i = oi; }
    }
  }
}

// Record of one (row, chunk) item: per segment its maximum (-inf when empty)
// and sum of exp(x - maximum) (log-sum-exp calls only).
struct StreamRec {
  float m[kSegs];
  float s[kSegs];
};

// Workspace header of the streaming path (reset before every call).
struct StreamHdr {
  int status;   // nonzero: a wait ran out
  int claim;    // next unclaimed (row, chunk) item
};
constexpr size_t kStreamHdrBytes = 256;

// `status0` is 0 except when the caller's process plants a failure to test
// the failure path (TV_TEST_VOCAB_STATUS, read on the host).
__global__ void stream_hdr_clear_kernel(StreamHdr* hdr, int status0) {
  griddep_wait();
  griddep_release();
  hdr->status = status0;
  hdr->claim = 0;
}

// Largest bf16 of this lane's share of a 1024-element segment (16-byte
// words lane-interleaved; words at or past V count as -inf), compared as
// packed bf16 pairs.
__device__ __forceinline__ float seg_max_bf16(const uint8_t* p, int e_first, int V) {
  constexpr int NV = kSegLen / 8 / 32;   // 16-byte words per lane
  const int lane = threadIdx.x & 31;
  const uint32_t ninf = 0xff80ff80u;     // (-inf, -inf)
  __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&ninf);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e0 = e_first + (j * 32 + lane) * 8;
    uint4 w = make_uint4(ninf, ninf, ninf, ninf);
    if (e0 < V) w = *reinterpret_cast<const uint4*>(p + static_cast<size_t>((j * 32 + lane) * 16));
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&w.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.z),
                                     *reinterpret_cast<const __nv_bfloat162*>(&w.w));
    m = __hmax2(m, __hmax2(a, b));
  }
  return fmaxf(__low2float(m), __high2float(m));
}
// Elements of segment `seg` of a row visible to this lane: 4 (bf16) or 8
// (fp32) 16-byte vectors, lane-interleaved; entries at or past V become -inf.
template <typename T>
__device__ __forceinline__ void seg_values(const uint8_t* p, int e_first, int V, float* v) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  constexpr int NV = kSegLen / VEC / 32;   // vectors per lane
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e0 = e_first + (j * 32 + lane) * VEC;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (e0 < V) w = *reinterpret_cast<const uint4*>(p + static_cast<size_t>((j * 32 + lane) * VEC) * sizeof(T));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[8 * j + 2 * q] = e0 < V ? bf16_lo(ws[q]) : -INFINITY;
        v[8 * j + 2 * q + 1] = e0 < V ? bf16_hi(ws[q]) : -INFINITY;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[4 * j + q] = e0 < V ? __uint_as_float(ws[q]) : -INFINITY;
    }
  }
}
// element number of value t of this lane within its segment
template <typename T>
__device__ __forceinline__ int seg_elem(int t) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  return ((t / VEC) * 32 + static_cast<int>(threadIdx.x & 31)) * VEC + t % VEC;
}

constexpr int kMergeBuf = 64;   // candidates a row's merge ranks in shared memory
// Rows per merge CTA (one warp each): 4, or 8 for calls of 256 rows or more
// without the log-sum-exp.  The merge CTAs are placed while the stream
// finishes, beside whatever else is then being placed on the SMs (in a
// verification step, the attention kernel's CTAs, which cannot share an SM
// with a merge CTA at two per SM): eight rows per CTA put the merge on half
// as many SMs, which took the D-cut step from 141.8 to 138.6 us, at about
// 1 us more for the call alone.
constexpr int kMergeWarpsMax = 8;
inline int merge_warps(int rows, bool lse) { return !lse && rows >= 256 ? 8 : 4; }

// Merge of one row by one warp: row max and log-sum-exp from the segment
// records; tau = the KMAX-th largest segment maximum; the segments whose
// maximum reaches tau are read again (two at a time, so that their loads
// overlap) and their elements >= tau ranked.
template <typename T, int KMAX, bool LSE>
__device__ __noinline__ void merge_row(const StreamRec* __restrict__ rec, int n_chunks, const T* __restrict__ x,
                                       int V, int dst, int k, int32_t* __restrict__ argmax,
                                       int32_t* __restrict__ topk_idx, float* __restrict__ topk_val,
                                       float* __restrict__ row_max, float* __restrict__ row_lse, float* s_bv,
                                       int* s_bi) {
  constexpr int SPL = kMaxFastSegs / 32;   // segment maxima per lane
  constexpr int EPS = kSegLen / 32;        // elements per lane per segment
  const int lane = threadIdx.x & 31;
  const int nseg = n_chunks * kSegs;
  const bool fast = nseg <= kMaxFastSegs;
  auto seg_first = [&](int g) { return (g / kSegs) * kVChunk + (g % kSegs) * kSegLen; };
  auto load_seg = [&](int g, float* v) {
    seg_values<T>(reinterpret_cast<const uint8_t*>(x + seg_first(g)), seg_first(g), V, v);
  };
  float M = -INFINITY, S = 0.f, tau = -INFINITY;
  // segment q * 32 + lane of the row in slot q
  float sm[SPL];
  if (fast) {
    float ss[SPL];
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
      const int g = q * 32 + lane;
      sm[q] = g < nseg ? __ldcg(&rec[g / kSegs].m[g % kSegs]) : -INFINITY;
      ss[q] = (LSE && g < nseg) ? __ldcg(&rec[g / kSegs].s[g % kSegs]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < SPL; ++q) M = fmaxf(M, sm[q]);
    M = redux_max(M);
    if constexpr (LSE) {
#pragma unroll
      for (int q = 0; q < SPL; ++q)
        if (sm[q] != -INFINITY) S += ss[q] * ex2((sm[q] - M) * kLog2e);
      S = warp_sum(S);
    }
    // tau: the KMAX-th largest segment maximum (-inf with fewer finite segments)
    float w[SPL];
#pragma unroll
    for (int q = 0; q < SPL; ++q) w[q] = sm[q];
    for (int t = 0; t < KMAX; ++t) {
      float mine = w[0];
#pragma unroll
      for (int q = 1; q < SPL; ++q) mine = fmaxf(mine, w[q]);
      const float b = redux_max(mine);
      tau = b;
      const unsigned hit = __ballot_sync(0xffffffffu, mine == b);
      if (lane == __ffs(hit) - 1) {   // drop one instance of b from this lane
        bool done = false;
#pragma unroll
        for (int q = 0; q < SPL; ++q)
          if (!done && w[q] == b) { w[q] = -INFINITY; done = true; }
      }
    }
  } else {
    for (int g = lane; g < nseg; g += 32) M = fmaxf(M, __ldcg(&rec[g / kSegs].m[g % kSegs]));
    M = redux_max(M);
    if constexpr (LSE) {
      for (int g = lane; g < nseg; g += 32) {
        const float m = __ldcg(&rec[g / kSegs].m[g % kSegs]);
        if (m != -INFINITY) S += __ldcg(&rec[g / kSegs].s[g % kSegs]) * ex2((m - M) * kLog2e);
      }
      S = warp_sum(S);
    }
  }
  // candidates >= tau of the segments whose maximum reaches tau
  int nb = 0;
  bool overflow = !fast;   // too many segments to select among: rank every element
  auto append = [&](const float* v, int g) {
#pragma unroll
    for (int t = 0; t < EPS; ++t) {
      const bool keep = v[t] >= tau && v[t] != -INFINITY;
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (bal) {
        const int pos = nb + __popc(bal & ((1u << lane) - 1u));
        if (keep && pos < kMergeBuf) { s_bv[pos] = v[t]; s_bi[pos] = seg_first(g) + seg_elem<T>(t); }
        nb += __popc(bal);
      }
    }
  };
  if (fast) {
    int pend = -1;   // a selected segment waiting for a partner
#pragma unroll 1
    for (int q = 0; q < SPL && !overflow; ++q) {
      unsigned sel = __ballot_sync(0xffffffffu, sm[q] != -INFINITY && sm[q] >= tau);
      while (sel && !overflow) {
        const int g = q * 32 + __ffs(sel) - 1;
        sel &= sel - 1u;
        if (pend < 0) {
          pend = g;
          continue;
        }
        float v0[EPS], v1[EPS];
        load_seg(pend, v0);
        load_seg(g, v1);
        append(v0, pend);
        append(v1, g);
        pend = -1;
        overflow = nb > kMergeBuf;
      }
    }
    if (pend >= 0 && !overflow) {
      float v0[EPS];
      load_seg(pend, v0);
      append(v0, pend);
      overflow = nb > kMergeBuf;
    }
  }
  __syncwarp();
  float ov[KMAX];
  int oi[KMAX];
  if (!overflow && nb <= 32) {
    float v = lane < nb ? s_bv[lane] : -INFINITY;
    int i = lane < nb ? s_bi[lane] : INT32_MAX;
    warp_bitonic_desc(v, i);
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
      ov[q] = __shfl_sync(0xffffffffu, v, q);
      oi[q] = __shfl_sync(0xffffffffu, i, q);
    }
  } else {
    // per-lane sorted lists, then KMAX rounds of warp merging: over the
    // buffer, or (heavy ties) over every element of every segment that can
    // hold a candidate
    float lv[KMAX];
    int li[KMAX];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) { lv[q] = -INFINITY; li[q] = INT32_MAX; }
    if (!overflow) {
      for (int t = lane; t < nb; t += 32) list_insert<KMAX>(lv, li, s_bv[t], s_bi[t]);
    } else {
      for (int g = 0; g < nseg; ++g) {
        const float m = __ldcg(&rec[g / kSegs].m[g % kSegs]);
        if (m == -INFINITY || m < tau) continue;
        float v[EPS];
        load_seg(g, v);
#pragma unroll
        for (int t = 0; t < EPS; ++t)
          if (v[t] != -INFINITY) list_insert<KMAX>(lv, li, v[t], seg_first(g) + seg_elem<T>(t));
      }
    }
    warp_merge_lists<KMAX>(lv, li, ov, oi);
  }
  if (lane == 0) {
    argmax[dst] = oi[0];
    if (row_max) row_max[dst] = M;
    if (LSE && row_lse) row_lse[dst] = M + logf(S);
  }
  if (k > 0 && lane < k) {
    float val = ov[0];
    int idx = oi[0];
#pragma unroll
    for (int q = 1; q < KMAX; ++q)
      if (lane == q) { val = ov[q]; idx = oi[q]; }
    if (topk_idx) topk_idx[static_cast<int64_t>(dst) * k + lane] = idx;
    if (topk_val) topk_val[static_cast<int64_t>(dst) * k + lane] = val;
  }
}

// Failure outputs of one row (a bounded wait ran out somewhere in the grid).
__device__ __forceinline__ void fail_row(int dst, int k, int32_t* argmax, int32_t* topk_idx, float* topk_val,
                                         float* row_max, float* row_lse, int lane) {
  const float nan = __int_as_float(0x7fc00000);
  if (lane == 0) {
    argmax[dst] = -1;
    if (row_max) row_max[dst] = nan;
    if (row_lse) row_lse[dst] = nan;
  }
  if (lane < k) {
    if (topk_idx) topk_idx[static_cast<int64_t>(dst) * k + lane] = -1;
    if (topk_val) topk_val[static_cast<int64_t>(dst) * k + lane] = nan;
  }
}

constexpr int kStreamThreads = kVThreads + 32;   // 8 compute warps + 1 producer warp

template <typename T, bool LSE>
__global__ void __launch_bounds__(kStreamThreads, 4) vocab_stream_kernel(
    const T* __restrict__ logits, int V, int64_t ld, const int32_t* __restrict__ row_idx, int rows, int n_chunks,
    StreamRec* __restrict__ rec, StreamHdr* __restrict__ hdr) {
  constexpr int EPT = kSegLen / 32;                        // values per lane per chunk
  constexpr int NW = kSegs;
  constexpr int S = stream_stages<T>();
  constexpr int kSChunkBytes = stream_chunk_bytes<T>();
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ int s_item[S], s_chunk[S];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int items = rows * n_chunks;          // < 2^31: rows <= 65535, chunks <= 2^15
  griddep_wait();
  griddep_release();
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sm_u32(&full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sm_u32(&empty[s])), "r"(NW) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == NW) {   // ------------------------------------------------ producer
    if (lane != 0) return;
    // two claims in flight: the item for this slot and the next one
    int a0 = atomicAdd(&hdr->claim, 1);
    int a1 = a0 < items ? atomicAdd(&hdr->claim, 1) : items;
    for (int q = 0;; ++q) {
      const int s = q % S;
      const int item = a0;
      a0 = a1;
      if (a1 < items) a1 = atomicAdd(&hdr->claim, 1);
      if (q >= S && !bar_wait_fast(sm_u32(&empty[s]), ((q / S) - 1) & 1)) {
        atomicExch(&hdr->status, 1);
        return;   // compute warps waiting on this slot time out in turn
      }
      if (item >= items) {   // no more work: an empty slot tells the compute warps
        s_item[s] = -1;
        bar_arrive_plain(sm_u32(&full[s]));
        return;
      }
      const int row = item / n_chunks, c = item - row * n_chunks;
      const int src = row_idx ? row_idx[row] : row;
      s_item[s] = item;
      s_chunk[s] = c;
      const int n = min(kVChunk, V - c * kVChunk);
      bulk_g2s(sm_u32(ring + s * kSChunkBytes),
               logits + static_cast<int64_t>(src) * ld + static_cast<int64_t>(c) * kVChunk,
               static_cast<uint32_t>(n * sizeof(T)), sm_u32(&full[s]));
    }
  }

  // ------------------------------------------------------------- compute warps
  for (int it = 0;; ++it) {
    const int s = it % S;
    if (!bar_wait_fast(sm_u32(&full[s]), (it / S) & 1)) {
      if (lane == 0) atomicExch(&hdr->status, 1);
      return;
    }
    const int item = s_item[s];
    if (item < 0) return;
    const int c = s_chunk[s];
    const int e_first = c * kVChunk + warp * kSegLen;
    const uint8_t* seg = ring + s * kSChunkBytes + static_cast<size_t>(warp) * kSegLen * sizeof(T);
    float wmax, wsum = 0.f;
    if constexpr (sizeof(T) == 2 && !LSE) {
      // maximum only: packed bf16 pairs straight from the ring, no unpacking
      wmax = redux_max(seg_max_bf16(seg, e_first, V));
      __syncwarp();
      if (lane == 0) bar_arrive_plain(sm_u32(&empty[s]));   // this warp is done with the slot
    } else {
      float v[EPT];
      seg_values<T>(seg, e_first, V, v);
      __syncwarp();
      if (lane == 0) bar_arrive_plain(sm_u32(&empty[s]));   // this warp is done with the slot
      float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int t = 4; t < EPT; ++t) m4[t & 3] = fmaxf(m4[t & 3], v[t]);
      wmax = redux_max(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
      if constexpr (LSE) {
        if (wmax != -INFINITY) {
          const float mb = wmax * kLog2e;
#pragma unroll
          for (int t = 0; t < EPT; ++t) wsum += ex2(fmaf(v[t], kLog2e, -mb));
        }
        wsum = warp_sum(wsum);
      }
    }
    if (lane == 0) {
      StreamRec* r = rec + item;
      r->m[warp] = wmax;
      r->s[warp] = wsum;
    }
  }
}

// One warp per row, after the stream: merge the row from its segment
// records, or, if a wait of the stream ran out, report failure on the row.
template <typename T, int KMAX, bool LSE>
__global__ void __launch_bounds__(32 * kMergeWarpsMax) vocab_stream_merge_kernel(
    const StreamRec* __restrict__ rec, int n_chunks, int rows, const T* __restrict__ logits, int V, int64_t ld,
    const int32_t* __restrict__ row_idx, int k, int32_t* __restrict__ argmax, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_val, float* __restrict__ row_max, float* __restrict__ row_lse,
    const StreamHdr* __restrict__ hdr) {
  __shared__ float s_bv[kMergeWarpsMax][kMergeBuf];
  __shared__ int s_bi[kMergeWarpsMax][kMergeBuf];
  griddep_wait();
  griddep_release();
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int row = blockIdx.x * (blockDim.x >> 5) + wl;
  if (row >= rows) return;
  const int src = row_idx ? row_idx[row] : row;
  if (__ldcg(&hdr->status) != 0) {
    // a bounded wait of the streaming kernel ran out: its records are
    // incomplete, so every row reports failure instead of a stale merge
    fail_row(src, k, argmax, topk_idx, topk_val, row_max, LSE ? row_lse : nullptr, lane);
    return;
  }
  merge_row<T, KMAX, LSE>(rec + static_cast<int64_t>(row) * n_chunks, n_chunks,
                          logits + static_cast<int64_t>(src) * ld, V, src, k, argmax, topk_idx, topk_val, row_max,
                          row_lse, s_bv[wl], s_bi[wl]);
}


// True for page-locked host memory the device reads in place.
static bool host_resident(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

template <typename T, int KMAX, bool LSE>
int vocab_launch(const T* logits, int rows, int V, int64_t ld, const int32_t* row_idx, int k,
                 int32_t* argmax, int32_t* topk_idx, float* topk_val, float* row_max,
                 float* row_lse, void* ws, cudaStream_t st) {
  const int n_chunks = (V + kVChunk - 1) / kVChunk;
  const bool vec_ok = aligned(logits, 16) && ((ld * static_cast<int64_t>(sizeof(T))) % 16 == 0);
  auto* part = reinterpret_cast<VocabPart<KMAX>*>(ws);
  // the streaming kernel's bulk copies need 16-byte rows and chunk tails; rows
  // of one chunk are reduced whole by one CTA each (the partial kernels below)
  const bool stream_ok = vec_ok && (static_cast<int64_t>(V) * sizeof(T)) % 16 == 0 && n_chunks > 1;
  if (stream_ok) {
    constexpr int smem = stream_stages<T>() * stream_chunk_bytes<T>();
    if (!smem_limit(vocab_stream_kernel<T, LSE>, smem)) return TV_ECUDA;
    const int items = rows * n_chunks;
    // Rows in page-locked host memory arrive over the host link, far slower
    // than HBM: a quarter of the SMs keep it busy and leave the rest to
    // kernels running beside this one.
    const int per_sm = sizeof(T) == 2 ? 4 : 2;   // shared memory: 3-slot rings of 16 KB / 32 KB chunks
    const int grid = std::min(items, host_resident(logits) ? std::max(1, sm_count() / 4)
                                                           : per_sm * sm_count());
    auto* hdr = reinterpret_cast<StreamHdr*>(ws);
    auto* rec = reinterpret_cast<StreamRec*>(static_cast<uint8_t*>(ws) + kStreamHdrBytes);
    static const int planted = [] {
      const char* e = std::getenv("TV_TEST_VOCAB_STATUS");
      return e ? std::atoi(e) : 0;
    }();
    int rc = launch_pdl(stream_hdr_clear_kernel, dim3(1), dim3(1), 0, st, hdr, planted);
    if (rc == TV_OK)
      rc = launch_pdl(vocab_stream_kernel<T, LSE>, dim3(grid), dim3(kStreamThreads), smem, st, logits, V, ld,
                      row_idx, rows, n_chunks, rec, hdr);
    const int mw = merge_warps(rows, LSE);
    if (rc == TV_OK)
      rc = launch_pdl(vocab_stream_merge_kernel<T, KMAX, LSE>, dim3((rows + mw - 1) / mw), dim3(32 * mw), 0, st,
                      rec, n_chunks, rows, logits, V, ld, row_idx, k, argmax, topk_idx, topk_val, row_max, row_lse,
                      hdr);
    return rc;
  }
  dim3 g1(n_chunks, rows);
  vocab_partial_kernel<T, KMAX, LSE><<<g1, kVThreads, 0, st>>>(logits, V, ld, row_idx, vec_ok, part);
  const int wpb = 4;
  vocab_merge_kernel<KMAX, LSE><<<(rows + wpb - 1) / wpb, 32 * wpb, 0, st>>>(
      part, n_chunks, rows, row_idx, k, argmax, topk_idx, topk_val, row_max, row_lse);
  return launch_status();
}

template <typename T>
int vocab_dispatch(const T* logits, int rows, int V, int64_t ld, const int32_t* row_idx, int k,
                   int32_t* argmax, int32_t* topk_idx, float* topk_val, float* row_max,
                   float* row_lse, void* ws, cudaStream_t st) {
  const bool lse = row_lse != nullptr;
#define TV_VOCAB_CASE(KM)                                                                        \
  return lse ? vocab_launch<T, KM, true>(logits, rows, V, ld, row_idx, k, argmax, topk_idx,     \
                                         topk_val, row_max, row_lse, ws, st)                    \
             : vocab_launch<T, KM, false>(logits, rows, V, ld, row_idx, k, argmax, topk_idx,    \
                                          topk_val, row_max, row_lse, ws, st);
  if (k <= 1) { TV_VOCAB_CASE(1) }
  if (k <= 8) { TV_VOCAB_CASE(8) }
  TV_VOCAB_CASE(16)
#undef TV_VOCAB_CASE
}

}  // namespace tv

TV_API size_t vocab_argmax_topk_workspace_size(int rows, int V, int k) {
  if (rows <= 0 || V <= 0) return 0;
  const size_t n_chunks = (static_cast<size_t>(V) + tv::kVChunk - 1) / tv::kVChunk;
  const size_t kmax = k <= 1 ? 1 : (k <= 8 ? 8 : 16);
  // the larger of the two paths' needs: fallback chunk partials, or the
  // streaming header, row counters and per-chunk segment records
  const size_t part = 2 * sizeof(float) + kmax * (sizeof(float) + sizeof(int));
  const size_t fallback = static_cast<size_t>(rows) * n_chunks * part;
  const size_t stream = tv::kStreamHdrBytes + static_cast<size_t>(rows) * n_chunks * sizeof(tv::StreamRec);
  return std::max(fallback, stream);
}

TV_API int vocab_argmax_topk(const void* logits, int dtype, int rows, int V, int64_t ld,
                             const int32_t* row_idx, int k, int32_t* argmax, int32_t* topk_idx,
                             float* topk_val, float* row_max, float* row_lse, void* ws,
                             size_t ws_bytes, tv_stream_t stream) {
  if (rows < 0 || V <= 0 || k < 0 || ld < V) return TV_EINVAL;
  if (k > TV_MAX_TOPK) return TV_EUNSUPPORTED;
  if (k > V) return TV_EINVAL;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_EINVAL;
  if (rows == 0) return TV_OK;
  if (!logits || !argmax) return TV_EINVAL;
  if (k > 0 && !topk_idx && !topk_val) return TV_EINVAL;
  if (rows > 65535) return TV_EUNSUPPORTED;
  const size_t need = vocab_argmax_topk_workspace_size(rows, V, k);
  if (!ws || ws_bytes < need || !tv::aligned(ws, 16)) return TV_EWORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TV_BF16)
    return tv::vocab_dispatch(static_cast<const uint16_t*>(logits), rows, V, ld, row_idx, k, argmax,
                              topk_idx, topk_val, row_max, row_lse, ws, st);
  return tv::vocab_dispatch(static_cast<const float*>(logits), rows, V, ld, row_idx, k, argmax,
                            topk_idx, topk_val, row_max, row_lse, ws, st);
}

// ---------------------------------------------------------------------------
// vocab_argmax_topk_noalloc: the same reduction for callers that cannot
// allocate device memory.  Its chunk partials live in a fixed file-scope
// device array instead of a caller workspace.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;   // TV_NOALLOC_SCRATCH_BYTES
constexpr int kNoallocMaxDevices = 64;

// Loaded with the library on every GPU that uses it and kept until exit.
static __device__ __align__(256) unsigned char g_vocab_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kNoallocMaxDevices] = {};

// Device address of g_vocab_scratch on the current device, looked up once per
// device (host code only knows the symbol's host-side shadow, not its address).
void* scratch_address(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) {
    *status = TV_ECUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_vocab_scratch) != cudaSuccess || !p) {
      *status = TV_ECUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *status = TV_OK;
  return g_scratch_ptr[dev];
}

}  // namespace

TV_API int vocab_argmax_topk_noalloc(const void* logits, int dtype, int rows, int V, int64_t ld,
                                     const int32_t* row_idx, int k, int32_t* argmax,
                                     int32_t* topk_idx, float* topk_val, float* row_max,
                                     float* row_lse, tv_stream_t stream) {
  if (rows < 0 || V <= 0 || k < 0 || ld < V) return TV_EINVAL;
  if (k > TV_MAX_TOPK) return TV_EUNSUPPORTED;
  if (k > V) return TV_EINVAL;
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_EINVAL;
  if (rows == 0) return TV_OK;
  if (!logits || !argmax) return TV_EINVAL;
  if (k > 0 && !topk_idx && !topk_val) return TV_EINVAL;
  if (rows > 65535) return TV_EUNSUPPORTED;
  if (vocab_argmax_topk_workspace_size(rows, V, k) > kNoallocScratchBytes) return TV_EWORKSPACE;
  int st = TV_OK;
  void* scratch = scratch_address(&st);
  if (st != TV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TV_BF16)
    return tv::vocab_dispatch(static_cast<const uint16_t*>(logits), rows, V, ld, row_idx, k, argmax,
                              topk_idx, topk_val, row_max, row_lse, scratch, s);
  return tv::vocab_dispatch(static_cast<const float*>(logits), rows, V, ld, row_idx, k, argmax,
                            topk_idx, topk_val, row_max, row_lse, scratch, s);
}
