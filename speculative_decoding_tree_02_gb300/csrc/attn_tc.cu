// tree_verify_attn, tensor-core path (bf16, head_dim 128): tree-masked GQA
// attention on the 5th-generation tensor cores (Graft page §2 third gear;
// SpecOPD page §02 proposal-tree scoring with the ancestor mask).  A tile is
// a set of query rows = (nodes x the g query heads of one KV head).
//
// 64-row tiles (a request's nodes x heads fit in 64 rows: the D-cut chains):
// attn_tc_kernel<64>, one CTA = (request, KV head, tile, split of the prefix
// keys), two CTAs per SM, keys in blocks of 64:
//   warp 2   TMA producer: Q once, then K and V blocks into separate 2-stage
//            rings (cp.async.bulk.tensor, 128-byte swizzle): a K slot is
//            reused once S of its block is done, a V slot once PV is.
//   warp 3   MMA issuer (one thread, event loop): S = Q K^T into a
//            double-buffered TMEM accumulator (128 x 64 fp32), then O += P V
//            into a TMEM accumulator (128 x 128 fp32); tcgen05.commit
//            signals mbarriers.  Also owns the TMEM allocation (256 columns).
//   warps 0-1 softmax, one thread per query row (its TMEM lane): load S,
//            apply the ancestor/prefix mask in registers, online base-2
//            softmax with lazy rescaling (O is rescaled in TMEM only when the
//            running max grows by more than 2^8), write P as bf16 into shared
//            memory in the UMMA K-major layout, and finally normalise O.
//            A warp none of whose rows is a live query keeps the barrier
//            protocol but skips the TMEM loads and the arithmetic.
// P is double-buffered: the softmax of block j waits only for PV(j-2) (its
// buffer), and for PV(j-1) only in the rare block where O must be rescaled,
// so the tensor core and the softmax warps overlap across blocks.
// S for block j+1 is computed while the softmax warps work on block j.
//
// 128-row tiles: attn_tc128_kernel (below), keys in blocks of 128.
//
// Every wait is bounded (2 s): on expiry the CTA records an error code in the
// workspace status word and stops; TMEM is always released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "attn.cuh"
#include "tc_common.cuh"

namespace tv {
namespace tc {

constexpr int kRows = 128;                   // MMA M: TMEM lanes
constexpr int kBlk = 64;                     // keys per block
constexpr int kD = 128;
constexpr uint32_t kKVHalf = 8192;           // 64 keys x 64 dims bf16


// Shared-memory layout for 64-row tiles.  The MMA always has M = 128: its
// rows 64..127 read the bytes that follow Q or P (still inside the CTA's
// shared memory) and the results of those rows are never used.  The layout
// is small enough for two CTAs per SM.
template <int LIVE>
struct Lay {
  static_assert(LIVE == 64, "128-row tiles run attn_tc128_kernel");
  // warp roles: softmax warps own TMEM lanes 32*(warp%4)..; only lanes 0..63
  // matter, so the CTA is 4 warps (softmax 0-1, TMA 2, MMA 3)
  static constexpr int kThreads = 128;
  static constexpr int kSoft = LIVE;                     // softmax threads
  static constexpr int kTmaWarp = 2;
  static constexpr int kMmaWarp = 3;
  static __device__ __forceinline__ bool soft_warp(int w) { return w < 2; }
  static constexpr int kStages = 2;                      // per ring (K and V)
  static constexpr uint32_t kQHalf = LIVE * 128;        // LIVE rows x 64 dims
  static constexpr uint32_t kPBytes = LIVE * 128;       // LIVE rows x 64 keys
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kPOff = 2 * kQHalf;         // two P buffers
  static constexpr uint32_t kKRingOff = kPOff + 2 * kPBytes;
  static constexpr uint32_t kVRingOff = kKRingOff + kStages * 2 * kKVHalf;
  static constexpr uint32_t kBarOff = kVRingOff + kStages * 2 * kKVHalf;
  static constexpr uint32_t kSmemBytes = kBarOff + 512 + 1024;   // barriers + 1 KB alignment slack
  static constexpr uint32_t kTmemSlot = kBarOff + 8 * 32;
  static constexpr uint32_t kAbortSlot = kTmemSlot + 4;
  static constexpr uint32_t kRedSlot = kTmemSlot + 8;   // [6 warps][3] ints (72 B)
  static_assert(kRedSlot + 72 <= kBarOff + 512, "barrier area");
  // TMEM (256 columns per CTA, two CTAs per SM): S0 | S1 | O; Q and P in
  // shared memory.
  static constexpr uint32_t kTmemCols = 256;
};

// mbarrier slots (8 bytes each) at kBarOff; K/V arrays sized for 5 stages
enum Bar { Q_FULL = 0, K_FULL = 1, V_FULL = 6, K_EMPTY = 11, V_EMPTY = 16, S_FULL = 21, S_FREE = 23,
           P_FULL = 25, P_FREE = 27, O_READY = 29, DRAIN = 30, N_BARS = 31 };

struct Maps {
  CUtensorMap q, kp, vp, kt, vt;
};

struct TcParams {
  Maps maps;
  AttnParams a;
  int* err;
};

// Merge of the pieces of one (request, KV head, tile), by the CTA of its last
// piece to finish: thread item = (query row, 32 output columns), pieces in
// order (weights 2^(m_i - M) l_i), so the result does not depend on which
// piece finished last.  All loads of up to four pieces are issued before any
// is used: one memory latency per item instead of one per piece.
template <int LIVE>
__device__ __forceinline__ void merge_pieces(const AttnParams& p, int r, int n0, int node_first, int cnt, int g,
                                             int kvh, int n_pieces, int nthreads) {
  constexpr int kGroup = 4;   // pieces whose loads are in flight together
  for (int item = threadIdx.x; item < LIVE * 4; item += nthreads) {
    const int rr = item >> 2, qd = item & 3;
    const int mln = node_first + rr / g;
    if (mln >= cnt) continue;
    const int mhead = kvh * g + rr % g;
    auto mslot = [&](int pc) {
      return (static_cast<int64_t>(pc) * p.B * p.max_nodes + static_cast<int64_t>(r) * p.max_nodes + mln) * p.Hq +
             mhead;
    };
    float M = -INFINITY;
    if (n_pieces > kGroup)
      for (int i = 0; i < n_pieces; ++i) M = fmaxf(M, __ldcg(&p.ws_ml[mslot(i)].x));
    float W = 0.f;
    float acc[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) acc[c] = 0.f;
    for (int i0 = 0; i0 < n_pieces; i0 += kGroup) {
      float2 ml[kGroup];
      float4 o4[kGroup][8];
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        ml[k] = make_float2(-INFINITY, 0.f);
        if (i0 + k < n_pieces) {
          ml[k] = __ldcg(&p.ws_ml[mslot(i0 + k)]);
          const float4* po = reinterpret_cast<const float4*>(p.ws_o + mslot(i0 + k) * kD + 32 * qd);
#pragma unroll
          for (int c = 0; c < 8; ++c) o4[k][c] = __ldcg(po + c);
        }
      }
      if (n_pieces <= kGroup) {
#pragma unroll
        for (int k = 0; k < kGroup; ++k) M = fmaxf(M, ml[k].x);
      }
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const float w = ml[k].y > 0.f ? ex2(ml[k].x - M) * ml[k].y : 0.f;   // empty piece: weight 0
        W += w;
        if (w == 0.f) continue;   // (an empty piece's o was never written)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          acc[4 * c] = fmaf(w, o4[k][c].x, acc[4 * c]);
          acc[4 * c + 1] = fmaf(w, o4[k][c].y, acc[4 * c + 1]);
          acc[4 * c + 2] = fmaf(w, o4[k][c].z, acc[4 * c + 2]);
          acc[4 * c + 3] = fmaf(w, o4[k][c].w, acc[4 * c + 3]);
        }
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint16_t* op = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(n0 + mln) * p.Hq + mhead) * kD + 32 * qd;
#pragma unroll
    for (int c = 0; c < 32; c += 8) {
      const uint4 v4 = make_uint4(pack_bf16(acc[c] * inv, acc[c + 1] * inv), pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv),
                                  pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv), pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv));
      *reinterpret_cast<uint4*>(op + c) = v4;
    }
    if (qd == 0 && p.lse)
      p.lse[static_cast<int64_t>(n0 + mln) * p.Hq + mhead] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------ kernel
// Smallest node index set in a node's ancestor mask (1 << 30 when empty):
// the mask words are read eight at a time, all loads of a batch in flight
// together, instead of one dependent load per word.
__device__ __forceinline__ int lowest_ancestor(const uint64_t* __restrict__ a, int words) {
  for (int w0 = 0; w0 < words; w0 += 8) {
    uint64_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = w0 + k < words ? a[w0 + k] : 0ull;
    int lo = 1 << 30;
#pragma unroll
    for (int k = 7; k >= 0; --k)
      if (v[k]) lo = (w0 + k) * 64 + __ffsll(static_cast<long long>(v[k])) - 1;
    if (lo != 1 << 30) return lo;
  }
  return 1 << 30;
}

template <int LIVE>
__global__ void __launch_bounds__(Lay<LIVE>::kThreads, 2) attn_tc_kernel(
    const __grid_constant__ TcParams P) {
  using L = Lay<LIVE>;
  constexpr int kThreads = L::kThreads;
  constexpr int kStages = L::kStages;
  constexpr uint32_t kQHalf = L::kQHalf, kPBytes = L::kPBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const AttnParams& p = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_release();
  const int kvh = blockIdx.x;
  const int4 unit = p.plan[static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y];   // plan order
  const int r = unit.x;
  if (r < 0) return;                                   // uniform: a unit without work
  const int piece = unit.y, n_pieces = unit.z, tile = unit.w;
  const int g = p.Hq / p.Hkv;
  const int nq = LIVE / g;
  const int n0 = p.node_off[r];
  const int N = p.node_off[r + 1] - n0;
  const int cnt = min(p.node_cnt ? min(p.node_cnt[r], N) : N, p.max_nodes);
  const int node_first = tile * nq;
  if (node_first >= cnt) return;                       // uniform: nothing to do
  const int pre0 = p.pre_off[r];
  const int Pr = p.pre_off[r + 1] - pre0;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbortSlot);
  int* red = reinterpret_cast<int*>(sm + L::kRedSlot);
  auto bar = [&](int i) { return sb + L::kBarOff + 8u * i; };

  // ---- row identity (softmax warps 2..5 own TMEM lanes 32*(warp%4) ..)
  const bool is_soft = L::soft_warp(warp);
  const int row = 32 * (warp & 3) + lane;
  const int ln = node_first + row / g;
  const int head = kvh * g + row % g;
  const bool active = is_soft && row < LIVE && ln < cnt;
  const int gn = n0 + ln;
  int vis = 0, lowest = 1 << 30;
  if (active) {
    vis = p.vis_prefix ? p.vis_prefix[gn] : Pr;
    vis = min(max(vis, 0), Pr);
    lowest = lowest_ancestor(p.anc + static_cast<int64_t>(gn) * p.anc_words, p.anc_words);
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
      if (i == S_FREE || i == S_FREE + 1 || i == P_FULL || i == P_FULL + 1) c = L::kSoft;
      mbar_init(bar(i), c);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == L::kMmaWarp) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + L::kTmemSlot),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + L::kTmemSlot);
  int vmax = 0, tlo = 1 << 30, thi = -1;
  for (int w = 0; w < kThreads / 32; ++w) {
    vmax = max(vmax, red[3 * w]);
    tlo = min(tlo, red[3 * w + 1]);
    thi = max(thi, red[3 * w + 2]);
  }

  // ---- key blocks of this CTA
  const int kb = piece * p.piece_len;
  const int ke = min(kb + p.piece_len, vmax);
  const int n_pre = ke > kb ? (ke - kb + kBlk - 1) / kBlk : 0;
  const bool do_tree = (piece == n_pieces - 1) && thi >= 0 && tlo <= thi;
  // partial-output slot of (piece, row)
  auto pslot = [&](int pc) {
    return (static_cast<int64_t>(pc) * p.B * p.max_nodes + static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
  };
  const int tb = do_tree ? (tlo & ~63) : 0;   // one 64-bit ancestor word per 64-key block
  const int n_tree = do_tree ? (thi + 1 - tb + kBlk - 1) / kBlk : 0;
  const int nblk = n_pre + n_tree;
  int* err = P.err;

  const uint32_t sQ = sb + L::kQOff, sP = sb + L::kPOff, sK = sb + L::kKRingOff, sV = sb + L::kVRingOff;
  const uint32_t tS0 = tmem, tO = tmem + 2 * kBlk;

  if (nblk > 0) {
    if (warp == L::kTmaWarp) {
      // ================= TMA producer (event loop: K and V rings refill independently)
      if (lane == 0) {
        mbar_expect_tx(bar(Q_FULL), 2 * kQHalf);
        tma_load_3d(sQ, &P.maps.q, 0, kvh * g, n0 + node_first, bar(Q_FULL));
        tma_load_3d(sQ + kQHalf, &P.maps.q, 64, kvh * g, n0 + node_first, bar(Q_FULL));
        // block j: its tensor maps and token coordinate
        auto where = [&](int j, const CUtensorMap*& mk, const CUtensorMap*& mv) {
          const bool tree = j >= n_pre;
          mk = tree ? &P.maps.kt : &P.maps.kp;
          mv = tree ? &P.maps.vt : &P.maps.vp;
          return tree ? n0 + tb + (j - n_pre) * kBlk : pre0 + kb + j * kBlk;
        };
        int nk = 0, nv = 0;
        uint64_t since = 0;
        while (nk < nblk || nv < nblk) {
          bool prog = false;
          if (nk < nblk && (nk < kStages || mbar_test(bar(K_EMPTY + nk % kStages), ((nk / kStages) - 1) & 1))) {
            const CUtensorMap *mk, *mv;
            const int coord = where(nk, mk, mv);
            const uint32_t dk = sK + (nk % kStages) * 2 * kKVHalf;
            mbar_expect_tx(bar(K_FULL + nk % kStages), 2 * kKVHalf);
            tma_load_3d(dk, mk, 0, kvh, coord, bar(K_FULL + nk % kStages));
            tma_load_3d(dk + kKVHalf, mk, 64, kvh, coord, bar(K_FULL + nk % kStages));
            ++nk;
            prog = true;
          }
          if (nv < nk && (nv < kStages || mbar_test(bar(V_EMPTY + nv % kStages), ((nv / kStages) - 1) & 1))) {
            const CUtensorMap *mk, *mv;
            const int coord = where(nv, mk, mv);
            const uint32_t dv = sV + (nv % kStages) * 2 * kKVHalf;
            mbar_expect_tx(bar(V_FULL + nv % kStages), 2 * kKVHalf);
            tma_load_3d(dv, mv, 0, kvh, coord, bar(V_FULL + nv % kStages));
            tma_load_3d(dv + kKVHalf, mv, 64, kvh, coord, bar(V_FULL + nv % kStages));
            ++nv;
            prog = true;
          }
          if (prog) since = 0;
          else if (!still_waiting(since, abort_flag, err, 1)) break;
        }
      }
    } else if (warp == L::kMmaWarp) {
      // ================= MMA issuer (event loop: S(j) as soon as its K and S
      // buffer are ready, PV(j) as soon as P(j) and V(j) are; neither waits
      // behind the other)
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(kRows, kBlk, 0);
        constexpr uint32_t idO = idesc_bf16(kRows, kD, 1);
        bool ok = mbar_wait(bar(Q_FULL), 0, abort_flag, err, 2);
        tc_fence_after();
        int ns = 0, npv = 0;
        uint64_t since = 0;
        while (ok && npv < nblk) {
          bool prog = false;
          // S buffer ns&1 is free once its previous S was read
          if (ns < nblk && mbar_test(bar(K_FULL + ns % kStages), (ns / kStages) & 1) &&
              (ns < 2 || mbar_test(bar(S_FREE + (ns & 1)), ((ns >> 1) - 1) & 1))) {
            tc_fence_after();
            const uint32_t kbase = sK + (ns % kStages) * 2 * kKVHalf;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t ko = (kk >> 2) * kKVHalf + (kk & 3) * 32;
              const uint32_t qo = (kk >> 2) * kQHalf + (kk & 3) * 32;
              umma_bf16(tS0 + kBlk * (ns & 1), sdesc(sQ + qo, 16, 1024), sdesc(kbase + ko, 16, 1024), idS, kk > 0);
            }
            umma_commit(bar(S_FULL + (ns & 1)));
            umma_commit(bar(K_EMPTY + ns % kStages));
            ++ns;
            prog = true;
          }
          if (npv < ns && mbar_test(bar(P_FULL + (npv & 1)), (npv >> 1) & 1) &&
              mbar_test(bar(V_FULL + npv % kStages), (npv / kStages) & 1)) {
            tc_fence_after();
            const uint32_t vbase = sV + (npv % kStages) * 2 * kKVHalf;
            const uint32_t pbase = sP + (npv & 1) * kPBytes;
#pragma unroll
            for (int kk = 0; kk < kBlk / 16; ++kk) {
              // P: K-major over the 64 keys (one 128-byte swizzle column); V:
              // MN-major, 16 keys = two 1 KB atoms, second 64-dim half kKVHalf
              // bytes away
              umma_bf16(tO, sdesc(pbase + kk * 32, 16, 1024), sdesc(vbase + kk * 2048, kKVHalf, 1024), idO,
                        (npv > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(bar(P_FREE + (npv & 1)));
            umma_commit(bar(O_READY));
            umma_commit(bar(V_EMPTY + npv % kStages));
            ++npv;
            prog = true;
          }
          if (prog) since = 0;
          else if (!still_waiting(since, abort_flag, err, 5)) ok = false;
        }
        // drain: every MMA issued above has completed before TMEM is released
        umma_commit(bar(DRAIN));
        mbar_wait(bar(DRAIN), 0, abort_flag, err, 7);
      }
    } else {
      // ================= softmax warps
      const float c2 = p.scale * kLog2e;
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const bool warp_live = __any_sync(0xffffffffu, active);
      uint8_t* prow = sm + L::kPOff + row * 128;
      if (!warp_live && row < LIVE) {
        // rows that are no live query: P stays zero in both buffers for the whole CTA
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          *reinterpret_cast<uint4*>(prow + (c8 << 4)) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(prow + kPBytes + (c8 << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        const int sb2 = j & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(S_FULL + sb2), (j >> 1) & 1, abort_flag, err, 8));
        if (!ok) break;
        tc_fence_after();
        uint32_t xr[2][32];
        if (warp_live) {
#pragma unroll
          for (int q = 0; q < 2; ++q) tmem_ld32(tS0 + kBlk * sb2 + lane_off + 32 * q, xr[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) pin(xr[q][c]);
        }
        tc_fence_before();
        mbar_arrive(bar(S_FREE + sb2));

        float corr = 1.f, rs = 0.f;
        bool rescale_row = false;
        uint32_t pk[2][16];
        if (warp_live) {
          // visibility of the 64 keys of block j for this row; full = all visible
          uint32_t vm[2] = {0u, 0u};
          if (active) {
            if (j < n_pre) {
              const int nv = min(vis, ke) - (kb + j * kBlk);
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int t = nv - 32 * q;
                vm[q] = t >= 32 ? 0xffffffffu : (t > 0 ? (1u << t) - 1u : 0u);
              }
            } else {
              const int w = (tb + (j - n_pre) * kBlk) >> 6;
              const uint64_t a0 = w < p.anc_words ? p.anc[static_cast<int64_t>(gn) * p.anc_words + w] : 0ull;
              vm[0] = static_cast<uint32_t>(a0);
              vm[1] = static_cast<uint32_t>(a0 >> 32);
            }
          }
          // raw scores; masked entries become -inf only in partial blocks
          if (__any_sync(0xffffffffu, (vm[0] & vm[1]) != 0xffffffffu)) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vm[q] >> c) & 1u)) xr[q][c] = __float_as_uint(-INFINITY);
          }
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(xr[q][c]));
          // running max in base-2 units of scale * q.k (scale > 0, so max commutes)
          const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
          const float mn = fmaxf(m, mloc);
          const bool grow = mn > m + 8.f;          // also true when m = -inf and mn is finite
          const float mu = grow ? mn : m;
          const float msafe = mu == -INFINITY ? 0.f : mu;
          float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float e0 = ex2(fmaf(__uint_as_float(xr[q][2 * c]), c2, -msafe));
              const float e1 = ex2(fmaf(__uint_as_float(xr[q][2 * c + 1]), c2, -msafe));
              sm4[c & 3] += e0 + e1;
              pk[q][c] = pack_bf16(e0, e1);
            }
          rs = (sm4[0] + sm4[1]) + (sm4[2] + sm4[3]);
          rescale_row = grow && m != -INFINITY;
          corr = rescale_row ? ex2(m - mu) : 1.f;
          m = mu;
        }
        // P buffer j&1 is free once PV(j-2) has completed.  O is touched only
        // when this warp must rescale: then PV(j-1) must have completed too.
        // Waits go in phase order so a parity wait is never two phases ahead.
        const bool need_o = warp_live && j > 0 && __any_sync(0xffffffffu, rescale_row);
        if (j >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(P_FREE + (j & 1)), ((j >> 1) - 1) & 1, abort_flag, err, 11));
          if (!ok) break;
        }
        if (need_o) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(O_READY), (j - 1) & 1, abort_flag, err, 9));
          if (!ok) break;
        }
        tc_fence_after();
        if (warp_live) {
          if (need_o) {
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
          // P row -> shared memory, K-major 128-byte swizzle (8 chunks of 8 keys)
          uint8_t* pdst = prow + (j & 1) * kPBytes;
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint32_t* src = &pk[c8 >> 2][(c8 & 3) * 4];
            *reinterpret_cast<uint4*>(pdst + ((c8 ^ (row & 7)) << 4)) = make_uint4(src[0], src[1], src[2], src[3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(bar(P_FULL + (j & 1)));
      }
      // all PV MMAs complete: the last two P buffers are released in order
      if (ok && nblk >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(P_FREE + ((nblk - 2) & 1)), ((nblk - 2) >> 1) & 1,
                                               abort_flag, err, 10));
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(P_FREE + ((nblk - 1) & 1)), ((nblk - 1) >> 1) & 1,
                                               abort_flag, err, 10));
      tc_fence_after();
      // ---- epilogue: O / l
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool write = active && ok;
      if (warp_live) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + 32 * q, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) pin(o[c]);
          if (write) {
            if (n_pieces == 1) {
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
              float* po = p.ws_o + pslot(piece) * kD + 32 * q;
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(po + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
            }
          }
        }
      }
      if (write) {
        if (n_pieces == 1) {
          if (p.lse) p.lse[static_cast<int64_t>(gn) * p.Hq + head] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        } else {
          p.ws_ml[pslot(piece)] = make_float2(m, l);
        }
      }
    }
  } else if (is_soft && active && n_pieces > 1) {
    // no keys in this piece: an empty partial
    p.ws_ml[pslot(piece)] = make_float2(-INFINITY, 0.f);
  }
  if (n_pieces > 1) __threadfence();   // this thread's partial, before the count below
  tc_fence_before();
  __syncthreads();
  // ---- pieces: the last of a (request, KV head, tile) to finish merges them
  int* last_flag = red;   // the reduction scratch is free again
  if (n_pieces > 1 && threadIdx.x == 0) {
    const int old = atomicAdd(&p.piece_cnt[(static_cast<int64_t>(r) * p.Hkv + kvh) * gridDim.y + tile], 1);
    *last_flag = old == n_pieces - 1;
  }
  if (n_pieces > 1) __syncthreads();
  if (warp == L::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::kTmemCols) : "memory");
  }
  if (n_pieces > 1 && *last_flag) {
    __threadfence();
    merge_pieces<LIVE>(p, r, n0, node_first, cnt, g, kvh, n_pieces, kThreads);
  }
}

// ------------------------------------------------------------------ 128-row tiles, 128-key blocks
// Tiles of 128 query rows (nodes x the group's heads) take keys in blocks of
// 128: S = Q K^T is one M = 128, N = 128 MMA per 16 dimensions (the N = 64
// shape costs the same issue time for half the keys), O += P V one M = 128,
// N = 128 MMA per 16 keys.  Tensor memory (512 columns): S0 | S1 | O | Q; Q
// and P are tensor-memory A operands, so the MMAs read only K and V from
// shared memory (rings of 3 K and 2 V blocks of 32 KB).
//   warp 0   TMA producer: Q once, then K and V blocks, each slot refilled
//            as soon as the MMA that read it has completed.
//   warp 1   MMA issuer (event loop): S(j) into buffer j & 1 once K(j) is in
//            and PV(j - 2) has completed (P(j - 2) lived in that buffer),
//            PV(j) once P(j) and V(j) are in; S(j + 1) runs while the
//            softmax warps work on block j.
//   warps 2-5 softmax, one thread per row (its TMEM lane): the 128 scores of
//            the block in registers, mask, online base-2 softmax with lazy
//            rescaling of O in tensor memory (only when the maximum grows by
//            more than 2^8; O must then be complete: PV(j - 1)), P as bf16
//            into the first 64 columns of S(j)'s buffer.
constexpr int kBlk2 = 128;                     // keys per block
constexpr uint32_t kHalf2 = kBlk2 * 128;       // 128 rows (keys or queries) x 64 dims bf16
struct Lay2 {
  static constexpr int kThreads = 192;
  static constexpr int kTmaWarp = 0, kMmaWarp = 1;
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr uint32_t kQOff = 0;                                   // Q staging: two halves
  static constexpr uint32_t kKOff = kQOff + 2 * kHalf2;                  // K ring
  static constexpr uint32_t kVOff = kKOff + kKStages * 2 * kHalf2;       // V ring
  static constexpr uint32_t kBarOff = kVOff + kVStages * 2 * kHalf2;
  static constexpr uint32_t kTmemSlot = kBarOff + 8 * 24;
  static constexpr uint32_t kAbortSlot = kTmemSlot + 4;
  static constexpr uint32_t kRedSlot = kTmemSlot + 8;                    // [6 warps][3] ints (72 B)
  static constexpr uint32_t kSmemBytes = kBarOff + 512 + 1024;
  static constexpr uint32_t kTmemCols = 512;                             // S0 | S1 | O | Q
  static_assert(kRedSlot + 72 <= kBarOff + 512, "barrier area");
};
// mbarrier slots: K_FULL/K_EMPTY per K stage, V_FULL/V_EMPTY per V stage,
// S_FULL/P_FULL/PV_DONE per S buffer
enum Bar2 { B2_Q = 0, B2_QT = 1, B2_K_FULL = 2, B2_K_EMPTY = 5, B2_V_FULL = 8, B2_V_EMPTY = 10, B2_S_FULL = 12,
            B2_P_FULL = 14, B2_PV_DONE = 16, B2_DRAIN = 18, B2_N = 19 };

__global__ void __launch_bounds__(Lay2::kThreads, 1) attn_tc128_kernel(const __grid_constant__ TcParams P) {
  using L = Lay2;
  constexpr int kThreads = L::kThreads;
  constexpr int LIVE = 128;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  const AttnParams& p = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_release();
  const int kvh = blockIdx.x;
  const int4 unit = p.plan[static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y];   // plan order
  const int r = unit.x;
  if (r < 0) return;                                   // uniform: a unit without work
  const int piece = unit.y, n_pieces = unit.z, tile = unit.w;
  const int g = p.Hq / p.Hkv;
  const int nq = LIVE / g;
  const int n0 = p.node_off[r];
  const int N = p.node_off[r + 1] - n0;
  const int cnt = min(p.node_cnt ? min(p.node_cnt[r], N) : N, p.max_nodes);
  const int node_first = tile * nq;
  if (node_first >= cnt) return;                       // uniform: nothing to do
  const int pre0 = p.pre_off[r];
  const int Pr = p.pre_off[r + 1] - pre0;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbortSlot);
  int* red = reinterpret_cast<int*>(sm + L::kRedSlot);
  auto bar = [&](int i) { return sb + L::kBarOff + 8u * i; };

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
    lowest = lowest_ancestor(p.anc + static_cast<int64_t>(gn) * p.anc_words, p.anc_words);
  }
  {
    const int vm = __reduce_max_sync(0xffffffffu, vis);
    const int lm = __reduce_min_sync(0xffffffffu, lowest);
    const int hm = __reduce_max_sync(0xffffffffu, active ? ln : -1);
    if (lane == 0) { red[3 * warp] = vm; red[3 * warp + 1] = lm; red[3 * warp + 2] = hm; }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < B2_N; ++i) {
      const bool soft_count = i == B2_QT || i == B2_P_FULL || i == B2_P_FULL + 1;
      mbar_init(bar(i), soft_count ? LIVE : 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == L::kMmaWarp) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + L::kTmemSlot),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + L::kTmemSlot);
  int vmax = 0, tlo = 1 << 30, thi = -1;
  for (int w = 0; w < kThreads / 32; ++w) {
    vmax = max(vmax, red[3 * w]);
    tlo = min(tlo, red[3 * w + 1]);
    thi = max(thi, red[3 * w + 2]);
  }

  // ---- key blocks of this CTA
  const int kb = piece * p.piece_len;
  const int ke = min(kb + p.piece_len, vmax);
  const int n_pre = ke > kb ? (ke - kb + kBlk2 - 1) / kBlk2 : 0;
  const bool do_tree = (piece == n_pieces - 1) && thi >= 0 && tlo <= thi;
  auto pslot = [&](int pc) {
    return (static_cast<int64_t>(pc) * p.B * p.max_nodes + static_cast<int64_t>(r) * p.max_nodes + ln) * p.Hq + head;
  };
  const int tb = do_tree ? (tlo & ~(kBlk2 - 1)) : 0;   // two 64-bit ancestor words per block
  const int n_tree = do_tree ? (thi + 1 - tb + kBlk2 - 1) / kBlk2 : 0;
  const int nblk = n_pre + n_tree;
  int* err = P.err;

  const uint32_t sQ = sb + L::kQOff, sK = sb + L::kKOff, sV = sb + L::kVOff;
  const uint32_t tS0 = tmem, tO = tmem + 2 * kBlk2, tQ = tmem + 2 * kBlk2 + kD;

  if (nblk > 0) {
    if (warp == L::kTmaWarp) {
      // ================= TMA producer: K and V rings refill independently
      if (lane == 0) {
        mbar_expect_tx(bar(B2_Q), 2 * kHalf2);
        tma_load_3d(sQ, &P.maps.q, 0, kvh * g, n0 + node_first, bar(B2_Q));
        tma_load_3d(sQ + kHalf2, &P.maps.q, 64, kvh * g, n0 + node_first, bar(B2_Q));
        auto where = [&](int j, const CUtensorMap*& mk, const CUtensorMap*& mv) {
          const bool tree = j >= n_pre;
          mk = tree ? &P.maps.kt : &P.maps.kp;
          mv = tree ? &P.maps.vt : &P.maps.vp;
          return tree ? n0 + tb + (j - n_pre) * kBlk2 : pre0 + kb + j * kBlk2;
        };
        int nk = 0, nv = 0;
        uint64_t since = 0;
        while (nk < nblk || nv < nblk) {
          bool prog = false;
          if (nk < nblk && (nk < KS || mbar_test(bar(B2_K_EMPTY + nk % KS), ((nk / KS) - 1) & 1))) {
            const CUtensorMap *mk, *mv;
            const int coord = where(nk, mk, mv);
            const uint32_t dk = sK + (nk % KS) * 2 * kHalf2;
            mbar_expect_tx(bar(B2_K_FULL + nk % KS), 2 * kHalf2);
            tma_load_3d(dk, mk, 0, kvh, coord, bar(B2_K_FULL + nk % KS));
            tma_load_3d(dk + kHalf2, mk, 64, kvh, coord, bar(B2_K_FULL + nk % KS));
            ++nk;
            prog = true;
          }
          if (nv < nk && (nv < VS || mbar_test(bar(B2_V_EMPTY + nv % VS), ((nv / VS) - 1) & 1))) {
            const CUtensorMap *mk, *mv;
            const int coord = where(nv, mk, mv);
            const uint32_t dv = sV + (nv % VS) * 2 * kHalf2;
            mbar_expect_tx(bar(B2_V_FULL + nv % VS), 2 * kHalf2);
            tma_load_3d(dv, mv, 0, kvh, coord, bar(B2_V_FULL + nv % VS));
            tma_load_3d(dv + kHalf2, mv, 64, kvh, coord, bar(B2_V_FULL + nv % VS));
            ++nv;
            prog = true;
          }
          if (prog) since = 0;
          else if (!still_waiting(since, abort_flag, err, 21)) break;
        }
      }
    } else if (warp == L::kMmaWarp) {
      // ================= MMA issuer (event loop)
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(kRows, kBlk2, 0);
        constexpr uint32_t idO = idesc_bf16(kRows, kD, 1);
        bool ok = mbar_wait(bar(B2_QT), 0, abort_flag, err, 22);
        tc_fence_after();
        int ns = 0, npv = 0;
        uint64_t since = 0;
        while (ok && npv < nblk) {
          bool prog = false;
          // S buffer ns & 1 is free once PV(ns - 2), which read P from it, has completed
          if (ns < nblk && mbar_test(bar(B2_K_FULL + ns % KS), (ns / KS) & 1) &&
              (ns < 2 || mbar_test(bar(B2_PV_DONE + (ns & 1)), ((ns >> 1) - 1) & 1))) {
            tc_fence_after();
            const uint32_t kbase = sK + (ns % KS) * 2 * kHalf2;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              umma_bf16_ts(tS0 + kBlk2 * (ns & 1), tQ + 8 * kk,
                           sdesc(kbase + (kk >> 2) * kHalf2 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
            umma_commit(bar(B2_S_FULL + (ns & 1)));
            umma_commit(bar(B2_K_EMPTY + ns % KS));
            ++ns;
            prog = true;
          }
          if (npv < ns && mbar_test(bar(B2_P_FULL + (npv & 1)), (npv >> 1) & 1) &&
              mbar_test(bar(B2_V_FULL + npv % VS), (npv / VS) & 1)) {
            tc_fence_after();
            const uint32_t vbase = sV + (npv % VS) * 2 * kHalf2;
#pragma unroll
            for (int kk = 0; kk < kBlk2 / 16; ++kk)
              umma_bf16_ts(tO, tS0 + kBlk2 * (npv & 1) + 8 * kk, sdesc(vbase + kk * 2048, kHalf2, 1024), idO,
                           (npv > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar(B2_PV_DONE + (npv & 1)));
            umma_commit(bar(B2_V_EMPTY + npv % VS));
            ++npv;
            prog = true;
          }
          if (prog) since = 0;
          else if (!still_waiting(since, abort_flag, err, 23)) ok = false;
        }
        // drain: every MMA issued above has completed before TMEM is released
        umma_commit(bar(B2_DRAIN));
        mbar_wait(bar(B2_DRAIN), 0, abort_flag, err, 24);
      }
    } else {
      // ================= softmax warps
      const float c2 = p.scale * kLog2e;
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const bool warp_live = __any_sync(0xffffffffu, active);
      // this row of Q -> tensor memory, dims (2c, 2c + 1) in column c: the
      // 128-byte swizzle puts 16-byte chunk c of a row at chunk c ^ (row & 7)
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B2_Q), 0, abort_flag, err, 25));
      if (ok && warp_live) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t qw[32];
          const uint8_t* src = sm + L::kQOff + h * kHalf2 + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
            qw[4 * c] = v.x; qw[4 * c + 1] = v.y; qw[4 * c + 2] = v.z; qw[4 * c + 3] = v.w;
          }
          tmem_st32(tQ + lane_off + 32 * h, qw);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(B2_QT));
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nblk && ok; ++j) {
        const int sb2 = j & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B2_S_FULL + sb2), (j >> 1) & 1, abort_flag, err, 26));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tS0 + kBlk2 * sb2;
        float rs = 0.f, corr = 1.f;
        bool rescale_row = false;
        uint32_t pw[64];
        if (warp_live) {
          uint32_t xr[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + lane_off + 32 * q, xr[q]);
          tmem_ld_wait();
          // visibility of the 128 keys of block j for this row (bit c of vm[q]: key 32q + c)
          uint32_t vm[4] = {0u, 0u, 0u, 0u};
          if (active) {
            if (j < n_pre) {
              const int nvis = min(vis, ke) - (kb + j * kBlk2);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int t = nvis - 32 * q;
                vm[q] = t >= 32 ? 0xffffffffu : (t > 0 ? (1u << t) - 1u : 0u);
              }
            } else {
              const int w = (tb + (j - n_pre) * kBlk2) >> 6;
              const int64_t a0 = static_cast<int64_t>(gn) * p.anc_words;
              const uint64_t a = w < p.anc_words ? p.anc[a0 + w] : 0ull;
              const uint64_t b = w + 1 < p.anc_words ? p.anc[a0 + w + 1] : 0ull;
              vm[0] = static_cast<uint32_t>(a);
              vm[1] = static_cast<uint32_t>(a >> 32);
              vm[2] = static_cast<uint32_t>(b);
              vm[3] = static_cast<uint32_t>(b >> 32);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) pin(xr[q][c]);
          // masked scores become -inf only in partial blocks
          if (__any_sync(0xffffffffu, (vm[0] & vm[1] & vm[2] & vm[3]) != 0xffffffffu)) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vm[q] >> c) & 1u)) xr[q][c] = __float_as_uint(-INFINITY);
          }
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(xr[q][c]));
          const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
          const float mn = fmaxf(m, mloc);
          const bool grow = mn > m + 8.f;          // also true when m = -inf and mn is finite
          const float mu = grow ? mn : m;
          const float msafe = mu == -INFINITY ? 0.f : mu;
          float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float e0 = ex2(fmaf(__uint_as_float(xr[q][2 * c]), c2, -msafe));
              const float e1 = ex2(fmaf(__uint_as_float(xr[q][2 * c + 1]), c2, -msafe));
              sm4[c & 3] += e0 + e1;
              pw[16 * q + c] = pack_bf16(e0, e1);
            }
          rs = (sm4[0] + sm4[1]) + (sm4[2] + sm4[3]);
          rescale_row = grow && m != -INFINITY;
          corr = rescale_row ? ex2(m - mu) : 1.f;
          m = mu;
        }
        // O is touched only when this warp must rescale: PV(j - 1) must then have completed
        if (warp_live && j > 0 && __any_sync(0xffffffffu, rescale_row)) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar(B2_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, err, 27));
          if (!ok) break;
          tc_fence_after();
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
        }
        if (warp_live) {
          l = l * corr + rs;
          // P row -> the first 64 columns of S(j)'s buffer (keys 2c, 2c + 1 in column c)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w16[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) w16[c] = pw[16 * q + c];
            tmem_st16(tS + lane_off + 16 * q, w16);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(bar(B2_P_FULL + sb2));
      }
      // the last PV has completed before O is read (PV(j) completes in order)
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B2_PV_DONE + ((nblk - 1) & 1)), ((nblk - 1) >> 1) & 1,
                                               abort_flag, err, 28));
      tc_fence_after();
      // ---- epilogue: O / l
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool write = active && ok;
      if (warp_live) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + 32 * q, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) pin(o[c]);
          if (write) {
            if (n_pieces == 1) {
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
              float* po = p.ws_o + pslot(piece) * kD + 32 * q;
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(po + c) =
                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
            }
          }
        }
      }
      if (write) {
        if (n_pieces == 1) {
          if (p.lse) p.lse[static_cast<int64_t>(gn) * p.Hq + head] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        } else {
          p.ws_ml[pslot(piece)] = make_float2(m, l);
        }
      }
    }
  } else if (is_soft && active && n_pieces > 1) {
    // no keys in this piece: an empty partial
    p.ws_ml[pslot(piece)] = make_float2(-INFINITY, 0.f);
  }
  if (n_pieces > 1) __threadfence();   // this thread's partial, before the count below
  tc_fence_before();
  __syncthreads();
  int* last_flag = red;   // the reduction scratch is free again
  if (n_pieces > 1 && threadIdx.x == 0) {
    const int old = atomicAdd(&p.piece_cnt[(static_cast<int64_t>(r) * p.Hkv + kvh) * gridDim.y + tile], 1);
    *last_flag = old == n_pieces - 1;
  }
  if (n_pieces > 1) __syncthreads();
  if (warp == L::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::kTmemCols) : "memory");
  }
  if (n_pieces > 1 && *last_flag) {
    __threadfence();
    merge_pieces<LIVE>(p, r, n0, node_first, cnt, g, kvh, n_pieces, kThreads);
  }
}

// Work plan (one CTA).  A unit is (request r, node tile t, piece): tile t
// of request r sees keys up to V_rt = the largest visible prefix among its
// nodes (the request's prefix without per-node prefixes) and takes
// n_rt = max(1, ceil(V_rt / piece_len)) pieces, the last of which also
// covers the tile's tree keys.  Units are placed in decreasing order of
// their prefix keys (64-key buckets; order within a bucket is free: the
// merge runs in piece order whatever the schedule), so the grid, which
// dispatches plan entries in order, runs the longest first.  Entries past
// the units have no work.  Also zeroes the status word and the piece
// counters.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 1024;
struct PlanArgs {
  const int32_t* pre_off;
  const int32_t* node_off;
  const int32_t* node_cnt;
  const int32_t* vis_prefix;
  int B, max_nodes, nq, tiles, piece_len, max_pieces, n_units, n_buckets;
  int4* plan;
  int* piece_cnt;
  int n_cnt;
  int* status;
};
__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(const PlanArgs a) {
  __shared__ int s_hist[kPlanBuckets], s_fill[kPlanBuckets];
  __shared__ int s_total;
  griddep_wait();
  griddep_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *a.status = 0;
  for (int i = tid; i < a.n_buckets; i += kPlanThreads) { s_hist[i] = 0; s_fill[i] = 0; }
  const int L = a.piece_len;
  const int pairs = a.B * a.tiles;   // <= n_cnt: the piece counters hold V_rt until the end
  int* vk_of = a.piece_cnt;
  // V_rt of every (request, tile), one warp per pair (-1: the tile has no nodes)
  for (int e = warp; e < pairs; e += kPlanThreads / 32) {
    const int r = e / a.tiles, t = e % a.tiles;
    const int n0 = a.node_off[r];
    const int N = a.node_off[r + 1] - n0;
    const int cnt = min(a.node_cnt ? min(a.node_cnt[r], N) : N, a.max_nodes);
    const int first = t * a.nq;
    const int Pr = a.pre_off[r + 1] - a.pre_off[r];
    int vk = Pr;
    if (a.vis_prefix) {
      vk = 0;
      for (int i = first + lane; i < min(first + a.nq, cnt); i += 32) vk = max(vk, min(max(a.vis_prefix[n0 + i], 0), Pr));
      vk = __reduce_max_sync(0xffffffffu, vk);
    }
    if (lane == 0) vk_of[e] = first < cnt ? vk : -1;
  }
  __syncthreads();
  auto pieces = [&](int vk) { return vk > 0 ? min((vk + L - 1) / L, a.max_pieces) : 1; };
  auto bucket = [&](int vk, int n, int pc) {
    const int keys = pc < n - 1 ? L : vk - (n - 1) * L;
    return min(a.n_buckets - 1, (keys + 63) / 64);
  };
  for (int e = tid; e < pairs; e += kPlanThreads) {
    const int vk = vk_of[e];
    if (vk < 0) continue;
    const int n = pieces(vk);
    for (int pc = 0; pc < n; ++pc) atomicAdd(&s_hist[bucket(vk, n, pc)], 1);
  }
  __syncthreads();
  // bucket starts in decreasing-length order (one warp, suffix sums)
  if (warp == 0) {
    int carry = 0;
    for (int b0 = a.n_buckets - 32; b0 >= 0; b0 -= 32) {
      const int b = b0 + 31 - lane;          // lane 0 takes the longest bucket of the group
      const int v = s_hist[b];
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      s_fill[b] = carry + x - v;             // units of longer buckets before this one
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_total = carry;
  }
  __syncthreads();
  for (int e = tid; e < pairs; e += kPlanThreads) {
    const int vk = vk_of[e];
    if (vk < 0) continue;
    const int n = pieces(vk);
    for (int pc = 0; pc < n; ++pc) {
      const int bk = bucket(vk, n, pc);
      const int pos = s_fill[bk] + atomicAdd(&s_hist[bk], -1) - 1;   // any slot of the bucket
      a.plan[pos] = make_int4(e / a.tiles, pc, n, e % a.tiles);
    }
  }
  for (int u = s_total + tid; u < a.n_units; u += kPlanThreads) a.plan[u] = make_int4(-1, 0, 0, 0);   // no work
  __syncthreads();
  for (int i = tid; i < a.n_cnt; i += kPlanThreads) a.piece_cnt[i] = 0;
}

// ------------------------------------------------------------------ host side
PlanArgs plan_args(const AttnParams& p, int nq, int tiles, int n_buckets, int* err) {
  PlanArgs a;
  a.pre_off = p.pre_off;
  a.node_off = p.node_off;
  a.node_cnt = p.node_cnt;
  a.vis_prefix = p.vis_prefix;
  a.B = p.B;
  a.max_nodes = p.max_nodes;
  a.nq = nq;
  a.tiles = tiles;
  a.piece_len = p.piece_len;
  a.max_pieces = p.n_units / (p.B * tiles);
  a.n_units = p.n_units;
  a.n_buckets = n_buckets;
  a.plan = const_cast<int4*>(p.plan);
  a.piece_cnt = p.piece_cnt;
  a.n_cnt = p.B * p.Hkv * tiles;
  a.status = err;
  return a;
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
  return g >= 1 && g <= 64 && (64 % g) == 0;
}

// 64 live rows when a whole request fits in one 64-row tile, else 128
static int tc_live(int max_nodes, int g) { return static_cast<long long>(max_nodes) * g <= 64 ? 64 : 128; }

void attn_tc_shape(int B, int max_nodes, int max_prefix, int Hq, int Hkv, int n_sm, int* piece_len,
                   int* max_pieces, int* tiles) {
  const int g = Hq / Hkv;
  const int live = tc_live(max_nodes, g);
  const int nq = live / g;
  *tiles = (max_nodes + nq - 1) / nq;
  // Units needed before requests are cut into pieces: 64-row tiles fill both
  // resident CTAs of an SM; 128-row tiles keep the tensor core of an SM busy
  // alone (the second resident CTA then overlaps their softmax).
  const long long slots = static_cast<long long>(n_sm) * (live == 64 ? 2 : 1);
  const int align = live == 64 ? 64 : 128;                       // keys per block
  // Enough (request, KV head, tile) units to fill the resident slots: whole
  // requests, longest first (a piece split costs a partial round trip and a
  // merge, more than the tail it removes).  Fewer: pieces sized so that the
  // units about fill the slots, but no shorter than 512 keys (64-row tiles)
  // or 2048 keys (128-row tiles, whose merge of 128 rows costs about as much
  // as 8 key blocks: one request of 61 nodes x 32 heads over a 2048-token
  // prefix took 29.7 us in four pieces, 28.2 in two and 26.3 in one; over
  // 8192 tokens 54.1 us in sixteen, 42.4 in four).
  const long long units = static_cast<long long>(B) * Hkv * *tiles;
  const long long min_piece = live == 64 ? 512 : 2048;
  long long L = std::max(align, (max_prefix + align - 1) / align * align);
  if (units < slots && max_prefix > min_piece) {
    const long long keys = units * max_prefix;
    L = std::max<long long>(min_piece, ((keys + slots - 1) / slots + align - 1) / align * align);
  }
  long long mp = max_prefix > 0 ? (max_prefix + L - 1) / L : 1;
  while (static_cast<long long>(B) * mp > 65535) {   // grid z limit
    L *= 2;
    mp = (max_prefix + L - 1) / L;
  }
  *piece_len = static_cast<int>(std::min<long long>(L, 1LL << 30));
  *max_pieces = static_cast<int>(std::max(1LL, mp));
}

template <int LIVE>
static int attn_tc_launch(const AttnParams& p, long long total_nodes, long long total_prefix, int* err,
                          cudaStream_t st) {
  using L = tc::Lay<LIVE>;
  if (!smem_limit(tc::attn_tc_kernel<LIVE>, static_cast<int>(L::kSmemBytes))) return TV_ECUDA;
  tc::TcParams P;
  std::memset(&P, 0, sizeof(P));
  P.a = p;
  P.err = err;
  const int g = p.Hq / p.Hkv;
  const int nq = LIVE / g;
  bool ok = tc::make_map(&P.maps.q, p.q, p.Hq, total_nodes, g, nq) &&
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
  const int tiles = (p.max_nodes + nq - 1) / nq;
  // 64-key length buckets up to the longest possible last piece, a multiple of 32
  const int n_buckets = static_cast<int>(std::min<long long>(
      tc::kPlanBuckets, (std::min<long long>(p.piece_len, p.max_prefix) / 64 + 2 + 31) / 32 * 32));
  int rc = launch_pdl(tc::attn_plan_kernel, dim3(1), dim3(tc::kPlanThreads), 0, st,
                      tc::plan_args(p, nq, tiles, n_buckets, err));
  if (rc != TV_OK) return rc;
  return launch_pdl(tc::attn_tc_kernel<LIVE>, dim3(p.Hkv, tiles, p.n_units / tiles), dim3(L::kThreads), L::kSmemBytes,
                    st, P);
}

// 128-row tiles: attn_tc128_kernel (128-key blocks, two CTAs per SM)
static int attn_tc128_launch(const AttnParams& p, long long total_nodes, long long total_prefix, int* err,
                             cudaStream_t st) {
  using L = tc::Lay2;
  if (!smem_limit(tc::attn_tc128_kernel, static_cast<int>(L::kSmemBytes))) return TV_ECUDA;
  tc::TcParams P;
  std::memset(&P, 0, sizeof(P));
  P.a = p;
  P.err = err;
  const int g = p.Hq / p.Hkv;
  const int nq = 128 / g;
  bool ok = tc::make_map(&P.maps.q, p.q, p.Hq, total_nodes, g, nq) &&
            tc::make_map(&P.maps.kt, p.k_tree, p.Hkv, total_nodes, 1, tc::kBlk2) &&
            tc::make_map(&P.maps.vt, p.v_tree, p.Hkv, total_nodes, 1, tc::kBlk2);
  if (ok && total_prefix > 0) {
    ok = tc::make_map(&P.maps.kp, p.k_pre, p.Hkv, total_prefix, 1, tc::kBlk2) &&
         tc::make_map(&P.maps.vp, p.v_pre, p.Hkv, total_prefix, 1, tc::kBlk2);
  } else if (ok) {
    P.maps.kp = P.maps.kt;   // never read: no prefix blocks exist
    P.maps.vp = P.maps.vt;
  }
  if (!ok) return TV_ECUDA;
  const int tiles = (p.max_nodes + nq - 1) / nq;
  const int n_buckets = static_cast<int>(std::min<long long>(
      tc::kPlanBuckets, (std::min<long long>(p.piece_len, p.max_prefix) / 64 + 2 + 31) / 32 * 32));
  int rc = launch_pdl(tc::attn_plan_kernel, dim3(1), dim3(tc::kPlanThreads), 0, st,
                      tc::plan_args(p, nq, tiles, n_buckets, err));
  if (rc != TV_OK) return rc;
  return launch_pdl(tc::attn_tc128_kernel, dim3(p.Hkv, tiles, p.n_units / tiles), dim3(L::kThreads), L::kSmemBytes,
                    st, P);
}

int attn_tc(const AttnParams& p, long long total_nodes, long long total_prefix, int* err, cudaStream_t st) {
  if (tc_live(p.max_nodes, p.Hq / p.Hkv) == 64) return attn_tc_launch<64>(p, total_nodes, total_prefix, err, st);
  return attn_tc128_launch(p, total_nodes, total_prefix, err, st);
}

}  // namespace tv
