// tree_verify_attn, tensor-core path (bf16, head_dim 128): tree-masked GQA
// attention on the 5th-generation tensor cores (Graft page §2 third gear;
// SpecOPD page §02 proposal-tree scoring with the ancestor mask).
//
// One CTA = (request, KV head, tile of 128 query rows = 128/g nodes x g heads,
// split of the prefix keys).  Keys stream in blocks of 128:
//   warp 0   TMA producer: Q once, then K and V blocks into a 2-stage ring
//            (cp.async.bulk.tensor, 128-byte swizzle).
//   warp 1   MMA issuer (one thread): S = Q K^T into a double-buffered TMEM
//            accumulator (128 x 128 fp32), then O += P V into a TMEM
//            accumulator (128 x 128 fp32); tcgen05.commit signals mbarriers.
//            Also owns the TMEM allocation.
//   warps 2-5 softmax, one thread per query row (its TMEM lane): load S,
//            apply the ancestor/prefix mask in registers, online base-2
//            softmax with lazy rescaling (O is rescaled in TMEM only when the
//            running max grows by more than 2^8), write P as bf16 into shared
//            memory in the UMMA K-major layout, and finally normalise O.
// S for block j+1 is computed while the softmax warps work on block j.
// Every wait is bounded (2 s): on expiry the CTA records an error code in the
// workspace status word and stops; TMEM is always released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "attn.cuh"

namespace tv {
namespace tc {

constexpr int kRows = 128;
constexpr int kBlk = 128;
constexpr int kD = 128;
constexpr int kThreads = 192;
constexpr uint32_t kHalf = 16384;            // one 64-column half of a 128 x 128 bf16 tile
constexpr uint32_t kTile = 2 * kHalf;        // 32 KB
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kQOff + kTile;    // 2 stages
constexpr uint32_t kVOff = kKOff + 2 * kTile;
constexpr uint32_t kPOff = kVOff + 2 * kTile;
constexpr uint32_t kBarOff = kPOff + kTile;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;   // barriers + 1 KB alignment slack
constexpr uint64_t kTimeoutNs = 2000000000ull;

// mbarrier slots (8 bytes each) at kBarOff
enum Bar { Q_FULL = 0, K_FULL = 1, V_FULL = 3, KV_EMPTY = 5, S_FULL = 7, S_FREE = 9, P_FULL = 11,
           O_READY = 12, DRAIN = 13, N_BARS = 14 };
constexpr uint32_t kTmemSlot = kBarOff + 8 * 16;
constexpr uint32_t kAbortSlot = kTmemSlot + 4;
constexpr uint32_t kRedSlot = kTmemSlot + 16;   // [6 warps][3] ints

struct Maps {
  CUtensorMap q, kp, vp, kt, vt;
};

struct TcParams {
  Maps maps;
  AttnParams a;
  int* err;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false on timeout (recorded) or when another role aborted.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* err, int code) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (gtime() - t0 > kTimeoutNs) break;
    }
  }
  *abort_flag = 1;
  if (err) atomicExch(err, code);
  return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define TV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                 "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : TV_R8(0), TV_R8(8), TV_R8(16), TV_R8(24)
      : "r"(taddr));
}
#undef TV_R8
#define TV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                 "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      TV_W8(0), TV_W8(8), TV_W8(16), TV_W8(24)
      : "memory");
}
#undef TV_W8
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Make register values produced by tcgen05.ld depend on the preceding wait.
__device__ __forceinline__ void pin(uint32_t& x) { asm volatile("" : "+r"(x)); }

// Shared-memory matrix descriptor: 128-byte swizzle, version field 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulate, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const AttnParams& p = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, tile = blockIdx.y;
  const int r = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int nq = kRows / g;
  const int n0 = p.node_off[r];
  const int N = p.node_off[r + 1] - n0;
  const int cnt = min(p.node_cnt ? min(p.node_cnt[r], N) : N, p.max_nodes);
  const int node_first = tile * nq;
  if (node_first >= cnt) return;                       // uniform: nothing to do
  const int pre0 = p.pre_off[r];
  const int Pr = p.pre_off[r + 1] - pre0;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kAbortSlot);
  int* red = reinterpret_cast<int*>(sm + kRedSlot);
  auto bar = [&](int i) { return sb + kBarOff + 8u * i; };

  // ---- row identity (softmax warps 2..5 own TMEM lanes 32*(warp%4) ..)
  const bool is_soft = warp >= 2;
  const int row = 32 * (warp & 3) + lane;
  const int ln = node_first + row / g;
  const int head = kvh * g + row % g;
  const bool active = is_soft && ln < cnt;
  const int gn = n0 + ln;
  int vis = 0, lowest = 1 << 30;
  if (active) {
    vis = p.vis_prefix ? p.vis_prefix[gn] : Pr;
    vis = min(max(vis, 0), Pr);
    for (int w = 0; w < p.anc_words; ++w) {
      const uint64_t a = p.anc[static_cast<int64_t>(gn) * p.anc_words + w];
      if (a) { lowest = w * 64 + __ffsll(static_cast<long long>(a)) - 1; break; }
    }
  }
  {
    const int vm = __reduce_max_sync(0xffffffffu, vis);
    const int lm = __reduce_min_sync(0xffffffffu, lowest);
    const int hm = __reduce_max_sync(0xffffffffu, active ? ln : -1);
    if (lane == 0) { red[3 * warp] = vm; red[3 * warp + 1] = lm; red[3 * warp + 2] = hm; }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < N_BARS; ++i) {
      uint32_t c = 1;
      if (i == S_FREE || i == S_FREE + 1 || i == P_FULL) c = kRows;
      mbar_init(bar(i), c);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + kTmemSlot),
                 "r"(512u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kTmemSlot);
  int vmax = 0, tlo = 1 << 30, thi = -1;
  for (int w = 0; w < kThreads / 32; ++w) {
    vmax = max(vmax, red[3 * w]);
    tlo = min(tlo, red[3 * w + 1]);
    thi = max(thi, red[3 * w + 2]);
  }

  // ---- key blocks of this CTA
  const int chunk = (p.max_prefix + p.n_split - 1) / p.n_split;
  const int kb = split * chunk;
  const int ke = min(kb + chunk, vmax);
  const int n_pre = ke > kb ? (ke - kb + kBlk - 1) / kBlk : 0;
  const bool do_tree = (split == p.n_split - 1) && thi >= 0 && tlo <= thi;
  const int tb = do_tree ? (tlo & ~63) : 0;
  const int n_tree = do_tree ? (thi + 1 - tb + kBlk - 1) / kBlk : 0;
  const int nblk = n_pre + n_tree;
  int* err = P.err;

  const uint32_t sQ = sb + kQOff, sK = sb + kKOff, sV = sb + kVOff, sP = sb + kPOff;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  if (nblk > 0) {
    if (warp == 0) {
      // ================= TMA producer
      if (lane == 0) {
        bool ok = true;
        mbar_expect_tx(bar(Q_FULL), kTile);
        tma_load_3d(sQ, &P.maps.q, 0, kvh * g, n0 + node_first, bar(Q_FULL));
        tma_load_3d(sQ + kHalf, &P.maps.q, 64, kvh * g, n0 + node_first, bar(Q_FULL));
        for (int j = 0; j < nblk && ok; ++j) {
          const int s = j & 1;
          if (j >= 2) ok = mbar_wait(bar(KV_EMPTY + s), ((j >> 1) - 1) & 1, abort_flag, err, 1);
          if (!ok) break;
          const bool tree = j >= n_pre;
          const int start = tree ? tb + (j - n_pre) * kBlk : kb + j * kBlk;
          const int coord = tree ? n0 + start : pre0 + start;
          const CUtensorMap* mk = tree ? &P.maps.kt : &P.maps.kp;
          const CUtensorMap* mv = tree ? &P.maps.vt : &P.maps.vp;
          const uint32_t dk = sK + s * kTile, dv = sV + s * kTile;
          mbar_expect_tx(bar(K_FULL + s), kTile);
          tma_load_3d(dk, mk, 0, kvh, coord, bar(K_FULL + s));
          tma_load_3d(dk + kHalf, mk, 64, kvh, coord, bar(K_FULL + s));
          mbar_expect_tx(bar(V_FULL + s), kTile);
          tma_load_3d(dv, mv, 0, kvh, coord, bar(V_FULL + s));
          tma_load_3d(dv + kHalf, mv, 64, kvh, coord, bar(V_FULL + s));
        }
      }
    } else if (warp == 1) {
      // ================= MMA issuer
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(kRows, kBlk, 0);
        constexpr uint32_t idO = idesc_bf16(kRows, kD, 1);
        bool ok = mbar_wait(bar(Q_FULL), 0, abort_flag, err, 2);
        tc_fence_after();
        auto issue_s = [&](int j) -> bool {
          const int s = j & 1;
          if (!mbar_wait(bar(K_FULL + s), (j >> 1) & 1, abort_flag, err, 3)) return false;
          if (j >= 2 && !mbar_wait(bar(S_FREE + s), ((j >> 1) - 1) & 1, abort_flag, err, 4)) return false;
          tc_fence_after();
          const uint32_t kbase = sK + s * kTile;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tS0 + 128 * s, sdesc(sQ + off, 16, 1024), sdesc(kbase + off, 16, 1024), idS, kk > 0);
          }
          umma_commit(bar(S_FULL + s));
          return true;
        };
        if (ok) ok = issue_s(0);
        if (ok && nblk > 1) ok = issue_s(1);
        for (int j = 0; j < nblk && ok; ++j) {
          const int s = j & 1;
          ok = mbar_wait(bar(P_FULL), j & 1, abort_flag, err, 5);
          if (ok) ok = mbar_wait(bar(V_FULL + s), (j >> 1) & 1, abort_flag, err, 6);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vbase = sV + s * kTile;
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;   // P: K-major over keys
            const uint32_t boff = kk * 2048;                            // V: 16 keys = 2 x 1 KB atoms
            umma_bf16(tO, sdesc(sP + aoff, 16, 1024), sdesc(vbase + boff, kHalf, 1024), idO,
                      (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar(O_READY));
          umma_commit(bar(KV_EMPTY + s));
          if (j + 2 < nblk) ok = issue_s(j + 2);
        }
        // drain: every MMA issued above has completed before TMEM is released
        umma_commit(bar(DRAIN));
        mbar_wait(bar(DRAIN), 0, abort_flag, err, 7);
      }
    } else {
      // ================= softmax warps
      const float c2 = p.scale * kLog2e;
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        const int s = j & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(S_FULL + s), (j >> 1) & 1, abort_flag, err, 8));
        if (!ok) break;
        tc_fence_after();
        uint32_t xr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS0 + 128 * s + lane_off + 32 * q, xr[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < 32; ++c) pin(xr[q][c]);
        tc_fence_before();
        mbar_arrive(bar(S_FREE + s));

        // visibility of the 128 keys of block j for this row
        uint32_t vm[4] = {0u, 0u, 0u, 0u};
        if (active) {
          if (j < n_pre) {
            const int start = kb + j * kBlk;
            const int nv = min(vis, ke) - start;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int t = nv - 32 * q;
              vm[q] = t >= 32 ? 0xffffffffu : (t > 0 ? (1u << t) - 1u : 0u);
            }
          } else {
            const int start = tb + (j - n_pre) * kBlk;
            const int w = start >> 6;
            const uint64_t a0 = w < p.anc_words ? p.anc[static_cast<int64_t>(gn) * p.anc_words + w] : 0ull;
            const uint64_t a1 = w + 1 < p.anc_words ? p.anc[static_cast<int64_t>(gn) * p.anc_words + w + 1] : 0ull;
            vm[0] = static_cast<uint32_t>(a0);
            vm[1] = static_cast<uint32_t>(a0 >> 32);
            vm[2] = static_cast<uint32_t>(a1);
            vm[3] = static_cast<uint32_t>(a1 >> 32);
          }
        }
        float mloc = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float x = ((vm[q] >> c) & 1u) ? __uint_as_float(xr[q][c]) * c2 : -INFINITY;
            xr[q][c] = __float_as_uint(x);
            mloc = fmaxf(mloc, x);
          }
        const float mn = fmaxf(m, mloc);
        const bool grow = mn > m + 8.f;          // also true when m = -inf and mn is finite
        const float mu = grow ? mn : m;
        const float msafe = mu == -INFINITY ? 0.f : mu;
        float rs = 0.f;
        uint32_t pk[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float e0 = ex2(__uint_as_float(xr[q][2 * c]) - msafe);
            const float e1 = ex2(__uint_as_float(xr[q][2 * c + 1]) - msafe);
            rs += e0 + e1;
            pk[q][c] = pack_bf16(e0, e1);
          }
        // P and O are free once PV of the previous block has completed
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(O_READY), (j - 1) & 1, abort_flag, err, 9));
          if (!ok) break;
          tc_fence_after();
        }
        const bool rescale_row = grow && m != -INFINITY;
        const float corr = rescale_row ? ex2(m - mu) : 1.f;
        if (__any_sync(0xffffffffu, rescale_row) && j > 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + 32 * q, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              pin(o[c]);
              o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
            }
            tmem_st32(tO + lane_off + 32 * q, o);
          }
          tmem_st_wait();
        }
        l = l * corr + rs;
        m = mu;
        // P row -> shared memory, K-major 128-byte swizzle: two 64-key halves
        uint8_t* prow = sm + kPOff + row * 128;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const int kh = ch >> 3, c8 = ch & 7;
          uint4 v4 = make_uint4(pk[ch >> 2][(ch & 3) * 4], pk[ch >> 2][(ch & 3) * 4 + 1],
                                pk[ch >> 2][(ch & 3) * 4 + 2], pk[ch >> 2][(ch & 3) * 4 + 3]);
          *reinterpret_cast<uint4*>(prow + kh * kHalf + ((c8 ^ (row & 7)) << 4)) = v4;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(bar(P_FULL));
      }
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(O_READY), (nblk - 1) & 1, abort_flag, err, 10));
        tc_fence_after();
      }
      // ---- epilogue: O / l
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool write = active && ok;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + 32 * q, o);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) pin(o[c]);
        if (write) {
          if (p.n_split == 1) {
            uint16_t* op = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(gn) * p.Hq + head) * kD + 32 * q;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 v4 = make_uint4(pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv),
                                    pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv),
                                    pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv),
                                    pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv));
              *reinterpret_cast<uint4*>(op + c) = v4;
            }
          } else {
            const int64_t slot = (static_cast<int64_t>(split) * p.B * p.max_nodes +
                                  static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
            float* po = p.ws_o + slot * kD + 32 * q;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(po + c) =
                  make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                              __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
          }
        }
      }
      if (write) {
        if (p.n_split == 1) {
          if (p.lse) p.lse[static_cast<int64_t>(gn) * p.Hq + head] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        } else {
          const int64_t slot = (static_cast<int64_t>(split) * p.B * p.max_nodes +
                                static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
          p.ws_ml[slot] = make_float2(m, l);
        }
      }
    }
  } else if (is_soft && active && p.n_split > 1) {
    // no keys in this split: an empty partial
    const int64_t slot = (static_cast<int64_t>(split) * p.B * p.max_nodes +
                          static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
    p.ws_ml[slot] = make_float2(-INFINITY, 0.f);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// [tokens, heads, 128] bf16 tensor; box = 64 dims x box_h heads x box_t tokens.
bool make_map(CUtensorMap* m, const void* base, int heads, long long tokens, int box_h, int box_t) {
  auto enc = encode_fn();
  if (!enc || tokens <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(heads) * kD * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_t)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool attn_tc_supported(int dtype, int d, int Hq, int Hkv) {
  if (dtype != TV_BF16 || d != tc::kD || Hq % Hkv) return false;
  const int g = Hq / Hkv;
  return g >= 1 && g <= 128 && (128 % g) == 0;
}

int attn_tc_splits(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm) {
  const int g = Hq / Hkv;
  const int nq = tc::kRows / g;
  const long long tiles = (max_nodes + nq - 1) / nq;
  const long long base = static_cast<long long>(B) * Hkv * tiles;
  long long s = (2LL * n_sm + base - 1) / base;
  s = std::min<long long>(s, std::max(1, (max_prefix + 511) / 512));
  return static_cast<int>(std::max(1LL, std::min(s, 64LL)));
}

int attn_tc(const AttnParams& p, long long total_nodes, long long total_prefix, int* err, cudaStream_t st) {
  static const bool attr_ok = cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(tc::kSmemBytes)) == cudaSuccess;
  if (!attr_ok) return TV_ECUDA;
  tc::TcParams P;
  std::memset(&P, 0, sizeof(P));
  P.a = p;
  P.err = err;
  const int g = p.Hq / p.Hkv;
  bool ok = tc::make_map(&P.maps.q, p.q, p.Hq, total_nodes, g, tc::kRows / g) &&
            tc::make_map(&P.maps.kt, p.k_tree, p.Hkv, total_nodes, 1, tc::kBlk) &&
            tc::make_map(&P.maps.vt, p.v_tree, p.Hkv, total_nodes, 1, tc::kBlk);
  if (ok && total_prefix > 0) {
    ok = tc::make_map(&P.maps.kp, p.k_pre, p.Hkv, total_prefix, 1, tc::kBlk) &&
         tc::make_map(&P.maps.vp, p.v_pre, p.Hkv, total_prefix, 1, tc::kBlk);
  } else if (ok) {
    P.maps.kp = P.maps.kt;   // never read: no prefix blocks exist
    P.maps.vp = P.maps.vt;
  }
  if (!ok) return TV_ECUDA;
  const int nq = tc::kRows / g;
  const int tiles = (p.max_nodes + nq - 1) / nq;
  dim3 grid(p.n_split, tiles, p.B * p.Hkv);
  tc::attn_tc_kernel<<<grid, tc::kThreads, tc::kSmemBytes, st>>>(P);
  if (p.n_split > 1) return attn_combine(p, st);
  return launch_status();
}

}  // namespace tv
