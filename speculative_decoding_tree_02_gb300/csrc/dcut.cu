// dcut_select: D-cut prefix-product scores and batch-global budget selection
// (D-cut page, technical summary §2 core mechanism and pipeline; §1 B x (D+1)).
//
// One CTA.  Scores are formed by one thread per request, strictly left to
// right in fp32 (no contraction: products only), so they equal the sequential
// definition bit for bit.  Each position's rank under (s desc, r asc, j asc)
// is a count over all T positions held in shared memory (T <= 8192); position
// t is kept for budget K iff rank(t) < K.  Packing offsets and indices follow
// from per-request counts, without assuming the kept set is a prefix.
#include <cmath>

#include "tv_common.cuh"

namespace tv {

constexpr int kDcutMaxPos = 8192;
constexpr int kDcutMaxRho = 8;

struct DcutK { int K[kDcutMaxRho]; };

__global__ void __launch_bounds__(1024) dcut_kernel(
    const float* __restrict__ conf, int B, int D, int n_rho, DcutK ks, float* __restrict__ score,
    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_len, int32_t* __restrict__ pack_off,
    int32_t* __restrict__ pack_idx) {
  extern __shared__ float s_sc[];                         // [T] scores
  int* s_rank = reinterpret_cast<int*>(s_sc + kDcutMaxPos);   // [T]
  const int N = D + 1;
  const int T = B * N;
  for (int r = threadIdx.x; r < B; r += blockDim.x) {
    float s = 1.f;
    s_sc[r * N] = s;
    score[static_cast<int64_t>(r) * N] = s;
    for (int j = 1; j <= D; ++j) {
      s = __fmul_rn(s, conf[static_cast<int64_t>(r) * D + j - 1]);
      s_sc[r * N + j] = s;
      score[static_cast<int64_t>(r) * N + j] = s;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float st = s_sc[t];
    int rank = 0;
    for (int u = 0; u < T; ++u) {
      const float su = s_sc[u];
      rank += (su > st) | ((su == st) & (u < t));
    }
    s_rank[t] = rank;
  }
  __syncthreads();
  for (int a = 0; a < n_rho; ++a) {
    const int K = ks.K[a];
    uint8_t* kp = keep + static_cast<int64_t>(a) * T;
    for (int t = threadIdx.x; t < T; t += blockDim.x) kp[t] = s_rank[t] < K;
    for (int r = threadIdx.x; r < B; r += blockDim.x) {
      int c = 0;
      for (int j = 0; j < N; ++j) c += s_rank[r * N + j] < K;
      keep_len[static_cast<int64_t>(a) * B + r] = c;
    }
  }
  __syncthreads();   // keep_len visible to the block
  if (pack_off || pack_idx) {
    if (threadIdx.x < n_rho) {
      const int a = threadIdx.x;
      int run = 0;
      for (int r = 0; r < B; ++r) {
        if (pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + r] = run;
        run += keep_len[static_cast<int64_t>(a) * B + r];
      }
      if (pack_off) pack_off[static_cast<int64_t>(a) * (B + 1) + B] = run;
    }
    __syncthreads();
    if (pack_idx) {
      for (int a = 0; a < n_rho; ++a) {
        const int K = ks.K[a];
        int32_t* pi = pack_idx + static_cast<int64_t>(a) * T;
        // packed slot of a kept (r, j): kept positions of earlier requests,
        // then kept positions of r before j
        for (int r = threadIdx.x; r < B; r += blockDim.x) {
          int o = 0;
          for (int r2 = 0; r2 < r; ++r2) o += keep_len[static_cast<int64_t>(a) * B + r2];
          for (int j = 0; j < N; ++j)
            if (s_rank[r * N + j] < K) pi[o++] = r * N + j;
        }
        for (int p = K + threadIdx.x; p < T; p += blockDim.x) pi[p] = -1;
      }
    }
  }
}

}  // namespace tv

TV_API size_t dcut_select_workspace_size(int B, int D, int n_rho) {
  (void)B; (void)D; (void)n_rho;
  return 0;
}

TV_API int dcut_select(const float* conf, int B, int D, const float* rho, int n_rho, float* score,
                       uint8_t* keep, int32_t* keep_len, int32_t* pack_off, int32_t* pack_idx,
                       void* ws, size_t ws_bytes, tv_stream_t stream) {
  (void)ws; (void)ws_bytes;
  if (B < 0 || D < 0 || n_rho < 0) return TV_EINVAL;
  if (B == 0 || n_rho == 0) return TV_OK;
  if (n_rho > tv::kDcutMaxRho) return TV_EUNSUPPORTED;
  const long long T = static_cast<long long>(B) * (D + 1);
  if (T > tv::kDcutMaxPos) return TV_EUNSUPPORTED;
  if (!conf && D > 0) return TV_EINVAL;
  if (!rho || !score || !keep || !keep_len) return TV_EINVAL;
  tv::DcutK ks{};
  for (int a = 0; a < n_rho; ++a) {
    const double r = static_cast<double>(rho[a]);   // host array
    if (!(r >= 0.0 && r <= 1.0)) return TV_EINVAL;
    ks.K[a] = static_cast<int>(std::floor(r * static_cast<double>(T) + 0.5));
  }
  static const int smem = [] {
    const int bytes = tv::kDcutMaxPos * (sizeof(float) + sizeof(int));
    cudaFuncSetAttribute(tv::dcut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return bytes;
  }();
  tv::dcut_kernel<<<1, 1024, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      conf, B, D, n_rho, ks, score, keep, keep_len, pack_off, pack_idx);
  return tv::launch_status();
}
