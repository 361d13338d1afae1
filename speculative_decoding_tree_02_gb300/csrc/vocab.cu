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
#include <float.h>

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

template <typename T, int KMAX, bool LSE>
int vocab_launch(const T* logits, int rows, int V, int64_t ld, const int32_t* row_idx, int k,
                 int32_t* argmax, int32_t* topk_idx, float* topk_val, float* row_max,
                 float* row_lse, void* ws, cudaStream_t st) {
  const int n_chunks = (V + kVChunk - 1) / kVChunk;
  const bool vec_ok = aligned(logits, 16) && ((ld * static_cast<int64_t>(sizeof(T))) % 16 == 0);
  auto* part = reinterpret_cast<VocabPart<KMAX>*>(ws);
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
  const size_t part = 2 * sizeof(float) + kmax * (sizeof(float) + sizeof(int));
  return static_cast<size_t>(rows) * n_chunks * part;
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

constexpr size_t kNoallocScratchBytes = size_t(8) << 20;   // TV_NOALLOC_SCRATCH_BYTES
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
