// Tree-masked attention on the 5th-generation tensor cores (tcgen05) of
// sm_103a: every flattened draft row attends the KV prefix and its own
// in-tree ancestors (EAGLE-2 article on sbmmt.com, attention-mask
// paragraph; EAGLE blog section 1.1: one target pass verifies the draft).
//
// One block per (KV split, KV head x 128-row tile, sequence), two blocks per
// SM, 8 warps each:
//   warps 0, 2 TMA producers: 64-key K tiles (warp 0) and V tiles (warp 2),
//              128-byte swizzle, each into its own 2-stage ring guarded by
//              mbarriers (expect-tx / commit); a K stage is released as soon
//              as its QK^T is done, a V stage after its P.V;
//   warp 1     owns 256 TMEM columns and issues tcgen05.mma:
//              S_j = Q K_j^T  (M=128, N=64, K=128)  into TMEM S (issued as
//              soon as the softmax has read S_{j-1} into registers),
//              O  += P_j V_j  (M=128, N=128, K=64, A = P_j read from TMEM);
//   warps 3-7  stage the Q tile (K-major, 128-byte swizzle) when it cannot
//              come by TMA (G not a divisor of 128);
//   warps 4-7  softmax, one thread per query row (= TMEM lane): mask by
//              prefix length / ancestor bits, online softmax in the log2
//              domain, P_j written to TMEM as bf16 pairs, lazy rescale of O
//              (only when the row max grows by more than 2^8).
// Two resident blocks per SM keep two independent pipelines in flight.  A
// 128-row tile packs (token, query head) rows of one KV head, so a GQA group
// shares every K/V tile.  The KV splits of one tile run as one thread-block
// cluster and merge their partial rows among themselves, each split a slice
// of the rows: a tile of at most 64 real rows (the MHA trees) moves them
// from TMEM straight into the owners' shared memory (distributed shared
// memory stores between two cluster barriers); larger tiles write them from
// TMEM to an L2-resident workspace and drop those lines after the merge
// (measured on GB300: merging in the last split to finish instead was about
// twice as slow, one SM reading every partial).  Every mbarrier wait is
// bounded: on expiry the block reports ET_DEV_TIMEOUT, stops, frees its TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "et_attn_internal.h"
#include "et_common.cuh"
#include "et_tc.cuh"

namespace et {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 2;                           // K ring and V ring, 2 tiles each (two blocks per SM)
constexpr uint32_t kHalfBytes = kTcKeys * 128;       // 64 rows x 128 B (64 of the 128 dims)
constexpr uint32_t kTileBytes = 2 * kHalfBytes;      // one K or V tile
constexpr uint32_t kQHalfBytes = kTcRows * 128;
constexpr uint32_t kQBytes = 2 * kQHalfBytes;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
constexpr uint32_t kOffMisc = kOffBar + 256;
// split merge through distributed shared memory (tiles of at most 64 real
// rows): the (max, sum) pairs received from every split; the rows land in
// the Q and K space
constexpr uint32_t kOffMlRecv = kOffMisc + 256;
constexpr int kDsmMaxRows = 64;     // real rows of a tile merged through DSMEM
constexpr int kDsmMaxSlots = 96;    // S * per for 2 <= S <= 16, per = ceil(rows / S) rounded up to even (<= 90)
constexpr uint32_t kMlRecvBytes = kDsmMaxSlots * 16;  // (max, sum, scale, -) per received row
constexpr uint32_t kSmemBytes = kOffMlRecv + kMlRecvBytes + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t kOffRecv = kOffQ;
constexpr uint32_t kRecvRowBytes = kTcDim * 2;  // a received row: 128 fp16 values scaled into [-1, 1]
static_assert(kDsmMaxSlots * kRecvRowBytes <= kOffV, "received rows fit the Q and K space");
// TMEM columns: S, O accumulator, P (bf16 pairs) double buffer
constexpr uint32_t kColS = 0, kColO = 64, kColP0 = 192, kColP1 = 224, kTmemCols = 256;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the row max grows by more than 2^8

// barrier slots
constexpr int B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_SFULL = 8, B_SFREE = 9, B_PFULL = 10,
              B_OFULL = 12, B_QFULL = 13, B_DRAIN = 14;
constexpr int kQWarps = 5;       // warps 3-7 stage Q
constexpr int kSoftmaxWarps = 4; // warps 4-7: one per TMEM lane quarter

// drop a 128-byte line of merge scratch from L2 without writing it back
__device__ __forceinline__ void discard_l2_line(const void *p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr uint32_t kIdescQK = idesc_bf16(kTcRows, kTcKeys, false);
constexpr uint32_t kIdescPV = idesc_bf16(kTcRows, kTcDim, true);

// 32 lanes x 32 bits x 16 columns (the narrow form of the TMEM loads in et_tc.cuh)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


__device__ __forceinline__ void split_range_tc(int L, int N, int S, int s, int &t0, int &t1, int &nP) {
  nP = (L + kTcKeys - 1) / kTcKeys;
  const int T = nP + (N + kTcKeys - 1) / kTcKeys;
  const int base = T / S, rem = T - base * S;  // split sizes differ by at most one tile
  t0 = s * base + min(s, rem);
  t1 = t0 + base + (s < rem ? 1 : 0);
}


// All lanes wait; the warp proceeds only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort, long long limit) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, limit));
}

// One warp: the sequence whose prefix is the blockIdx.z-th longest (ties:
// lower index first) into *seq, its first KV row into *row0.  B <= kLptMaxB.
__device__ __noinline__ void rank_by_prefix(const int *prefix_len, const long long *kv_row0, int B, int *s_len, int *seq,
                                            long long *row0) {
  const int lane = threadIdx.x & 31;
  for (int j = lane; j < B; j += 32) s_len[j] = prefix_len[j];
  __syncwarp();
  for (int c = lane; c < B; c += 32) {
    const int Lc = s_len[c];
    int rank = 0;
    for (int j = 0; j < B; ++j) {
      const int Lj = s_len[j];
      rank += (Lj > Lc || (Lj == Lc && j < c)) ? 1 : 0;
    }
    if (rank == (int)blockIdx.z) {
      *seq = c;
      *row0 = kv_row0 ? kv_row0[c] : 0;
    }
  }
}

// kLpt: a ragged batch of 2..kLptMaxB sequences goes out longest prefix
// first; the other instance keeps the grid order (and the registers the
// remapped index would hold)
template <bool kLpt>
__global__ void __launch_bounds__(kThreads, 2)
    k_attn_tc(const __grid_constant__ CUtensorMap tm_kp, const __grid_constant__ CUtensorMap tm_vp,
              const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
              const __grid_constant__ CUtensorMap tm_q, const TcLaunch a) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ int row_tok[kTcRows], row_head[kTcRows];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = saddr(sm);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc + 16);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8u * (uint32_t)i; };

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int s = blockIdx.x, g = blockIdx.y / a.MT, mt = blockIdx.y - g * a.MT;
  const int N = a.N;

  // Longest prefix first: blocks go out in grid order (sequence = z slowest),
  // so block z takes the sequence with the z-th longest prefix (ties: lower
  // index first) and the ragged batch's longest streams start in the first
  // wave instead of trailing the last one.  One warp ranks the lengths
  // (B <= 64; larger batches keep the grid order).
  __shared__ int s_len[kLptMaxB];
  __shared__ int s_seq;
  __shared__ long long s_row0;
  constexpr bool lpt = kLpt;
  // warp 2 ranks; the caller makes s_seq / s_row0 visible with a block barrier
  auto rank_sequences = [&]() { rank_by_prefix(a.prefix_len, a.kv_row0, a.B, s_len, &s_seq, &s_row0); };

  // with inputs_ready the prefix lengths and start rows are inputs: their
  // loads go out first and overlap the set-up
  int L_in = 0;
  long long row0_in = 0;
  if (a.inputs_ready) {
    if (lpt) {
      if (warp == 2) rank_sequences();
    } else {
      L_in = a.prefix_len[blockIdx.z];
      row0_in = a.kv_row0 ? a.kv_row0[blockIdx.z] : 0;
    }
  }
  // ---- set-up that touches no global memory (it overlaps the previous kernel's tail) ----
  if (warp == 3 && lane < 5) {  // the five tensor maps into the TMA descriptor cache
    prefetch_tmap(lane == 0 ? &tm_kp : lane == 1 ? &tm_vp : lane == 2 ? &tm_kt : lane == 3 ? &tm_vt : &tm_q);
  }
  if (t == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
      mbar_init(bar(B_PFULL + i), kSoftmaxWarps);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), kSoftmaxWarps);
    mbar_init(bar(B_OFULL), 1);
    mbar_init(bar(B_QFULL), a.q_tma ? 1 : kQWarps);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (t < kTcRows) {
    const int R = mt * kTcRows + t;
    const int i = R / a.G;
    row_tok[t] = i < N ? i : -1;
    row_head[t] = g * a.G + (R - i * a.G);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (!a.inputs_ready) {
    pdl_wait();     // the previous kernel in the stream has completed (the inputs may come from it)
    pdl_trigger();  // after the TMEM allocation: a waiting dependent block must not hold the TMEM this block needs
    if (lpt) {
      if (warp == 2) rank_sequences();
      __syncthreads();
    }
  }
  const int b = lpt ? s_seq : (int)blockIdx.z;  // lpt is a compile-time constant
  if (a.inputs_ready && lpt) {
    L_in = s_len[b];
    row0_in = s_row0;
  }
  // with inputs_ready the previous kernel writes none of Q, K/V or the prefix
  // lengths: the whole prefix streams before the wait; the softmax waits
  // before the first tree tile (the mask), every thread before the outputs
  const int L = a.inputs_ready ? L_in : a.prefix_len[b];
  const long long S_b = a.kv_head_stride > 0 ? a.kv_head_stride : L;
  const long long row0 = a.inputs_ready ? row0_in : (a.kv_row0 ? a.kv_row0[b] : 0);
  int t0, t1, nP;
  split_range_tc(L, N, a.S, s, t0, t1, nP);
  const int T = t1 - t0;
  if (t == 0) {
    // the first K and V tiles and the Q tile go out first: their round trip
    // is the longest latency of the prologue
    for (int j = 0; j < T && j < kStages; ++j) {
      const int tile = t0 + j;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t fb = bar((kv ? B_VFULL : B_KFULL) + j);
        mbar_expect_tx(fb, kTileBytes);
        const uint32_t dst = sb + (kv ? kOffV : kOffK) + j * kTileBytes;
        if (tile < nP) {
          const int row = (int)(row0 + (long long)g * S_b + (long long)tile * kTcKeys);
          tma_2d(dst, kv ? &tm_vp : &tm_kp, 0, row, fb);
          tma_2d(dst + kHalfBytes, kv ? &tm_vp : &tm_kp, 64, row, fb);
        } else {
          const int tr = b * N + (tile - nP) * kTcKeys;
          tma_3d(dst, kv ? &tm_vt : &tm_kt, 0, g, tr, fb);
          tma_3d(dst + kHalfBytes, kv ? &tm_vt : &tm_kt, 64, g, tr, fb);
        }
      }
    }
    if (a.q_tma && T > 0) {  // rows (token, head in group) of KV head g: one 4-D box per 64 dims
      const uint32_t qb = bar(B_QFULL);
      mbar_expect_tx(qb, kQBytes);
      const int tok0 = b * N + mt * (kTcRows / a.G);
      tma_4d(sb + kOffQ, &tm_q, 0, 0, g, tok0, qb);
      tma_4d(sb + kOffQ + kQHalfBytes, &tm_q, 64, 0, g, tok0, qb);
    }
  }
  if (t == 0 && L > 0 && row0 + (long long)g * S_b + L > a.kv_rows) flag_status(a.dev_status, ET_DEV_BAD_INDEX);

  if (warp == 0 || warp == 2) {
    // ---------------- TMA producers: warp 0 streams K tiles, warp 2 V tiles ----------------
    if (lane == 0 && T > 0) {
      const bool isK = warp == 0;
      const CUtensorMap *mp = isK ? &tm_kp : &tm_vp;
      const CUtensorMap *mt_ = isK ? &tm_kt : &tm_vt;
      const int bF = isK ? B_KFULL : B_VFULL, bE = isK ? B_KEMPTY : B_VEMPTY;
      const uint32_t base = sb + (isK ? kOffK : kOffV);
      int issued = T < kStages ? T : kStages;  // the first stages went out at the top
      for (int j = issued; j < T; ++j) {
        const int stage = j % kStages;
        if (j >= kStages && !mbar_wait(bar(bE + stage), (uint32_t)((j / kStages) - 1) & 1u, abort_flag, a.wait_cycles)) break;
        const uint32_t fb = bar(bF + stage);
        mbar_expect_tx(fb, kTileBytes);
        const uint32_t dst = base + stage * kTileBytes;
        const int tile = t0 + j;
        if (tile < nP) {
          const int row = (int)(row0 + (long long)g * S_b + (long long)tile * kTcKeys);
          tma_2d(dst, mp, 0, row, fb);
          tma_2d(dst + kHalfBytes, mp, 64, row, fb);
        } else {
          const int tr = b * N + (tile - nP) * kTcKeys;
          tma_3d(dst, mt_, 0, g, tr, fb);
          tma_3d(dst + kHalfBytes, mt_, 64, g, tr, fb);
        }
        issued = j + 1;
      }
      // do not leave while copies are in flight (the earlier stages were consumed)
      const int first = issued > kStages ? issued - kStages : 0;
      for (int j = first; j < issued; ++j) mbar_drain(bar(bF + j % kStages), (uint32_t)(j / kStages) & 1u);
      if (isK && a.q_tma) mbar_drain(bar(B_QFULL), 0);  // the Q tile this thread sent at the top, too
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && T > 0) {
      auto issue_s = [&](int j) {
        const int stage = j % kStages;
        const uint32_t kbase = sb + kOffK + stage * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTcDim / 16; ++kk) {
          const uint64_t ad = sw128_desc(sb + kOffQ + (kk >> 2) * kQHalfBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(kbase + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
          tc_mma(tmem + kColS, ad, bd, kIdescQK, kk > 0);
        }
        tc_commit(bar(B_SFULL));
        if (j + kStages < T) tc_commit(bar(B_KEMPTY + stage));  // K tile consumed once S_j is done
      };
      bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, a.wait_cycles) && mbar_wait(bar(B_KFULL + 0), 0, abort_flag, a.wait_cycles);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < T; ++j) {
        // S_{j+1} as soon as the softmax has read S_j out of TMEM
        if (j + 1 < T) {
          if (!mbar_wait(bar(B_SFREE), (uint32_t)j & 1u, abort_flag, a.wait_cycles)) break;
          if (!mbar_wait(bar(B_KFULL + (j + 1) % kStages), (uint32_t)((j + 1) / kStages) & 1u, abort_flag, a.wait_cycles)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        const int stage = j % kStages;
        if (!mbar_wait(bar(B_PFULL + (j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, a.wait_cycles)) break;
        if (!mbar_wait(bar(B_VFULL + stage), (uint32_t)(j / kStages) & 1u, abort_flag, a.wait_cycles)) break;
        tc_fence_after();
        const uint32_t pcol = tmem + ((j & 1) ? kColP1 : kColP0);
        const uint32_t vbase = sb + kOffV + stage * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk) {
          const uint64_t bd = sw128_desc(vbase + kk * 2048, kHalfBytes, 1024);
          tc_mma_ts(tmem + kColO, pcol + 8 * kk, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_OFULL));
        if (j + kStages < T) tc_commit(bar(B_VEMPTY + stage));
      }
      // every MMA this thread issued has finished before TMEM can be freed
      // (after an expired wait the softmax may not have waited for them)
      tc_commit(bar(B_DRAIN));
      mbar_drain(bar(B_DRAIN), 0);
    }
  }
  if (warp >= 3 && !a.q_tma) {
    // ---------------- Q tile -> shared memory (warps 3-7) when G does not divide 128 ----------------
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.q);
    for (int x = t - 96; x < kTcRows * 16; x += kThreads - 96) {
      const int r = x >> 4, c = x & 15;
      const int i = row_tok[r];
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (i >= 0)
        v = *reinterpret_cast<const uint4 *>(Q + (((long long)b * N + i) * a.Hq + row_head[r]) * kTcDim + c * 8);
      const uint32_t dst = sb + kOffQ + (uint32_t)(c >> 3) * kQHalfBytes + (uint32_t)r * 128u +
                           (uint32_t)(((c & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_QFULL));
  }

  // softmax: warp w (4..7) owns TMEM lane quarter w - 4 = tile rows 32 (w-4) .. +31
  const bool smx = warp >= 4;
  const int r = t - 128;
  float m_used = -INFINITY, l = 0.f;
  const int my_tok = smx ? row_tok[r] : -1;
  bool ok_rows = true;
  if (smx) {
    const bool active = __any_sync(0xffffffffu, my_tok >= 0);  // warp-uniform: any real row here
    unsigned long long mw0 = 0ull, mw1 = 0ull;
    // the mask comes from the previous kernel: read it after the programmatic
    // wait, at the top (without inputs_ready) or at the first tree tile
    const int j_mask = a.inputs_ready ? (nP > t0 ? nP - t0 : 0) : 0;
    const uint32_t lane_base = tmem + ((uint32_t)(r & ~31) << 16);
    const float scale = a.scale_log2;
    uint32_t raw[64];
    for (int j = 0; j < T; ++j) {
      const int tile = t0 + j;
      if (j == j_mask) {
        if (a.inputs_ready) pdl_wait();
        if (my_tok >= 0) {  // in flight while S of this tile completes
          mw0 = a.mask[((long long)b * N + my_tok) * a.W];
          if (a.W > 1) mw1 = a.mask[((long long)b * N + my_tok) * a.W + 1];
        }
      }
      if (!warp_wait(bar(B_SFULL), (uint32_t)j & 1u, abort_flag, a.wait_cycles)) { ok_rows = false; break; }
      tc_fence_after();
      if (active) {
        tmem_ld64(lane_base + kColS, raw);
        tmem_wait_ld();
      }
      // S is free for S_{j+1} as soon as it sits in registers
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE));
      if (active) {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        const int lim = tile < nP ? L - tile * kTcKeys : 0;
        if (tile < nP && lim >= kTcKeys) {  // a full prefix tile: nothing to mask
#pragma unroll
          for (int c = 0; c < 64; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(raw[c]));
        } else {
          // keep bits: the first lim keys of the partial prefix tile (0 < lim < 64), else the row's mask word
          const unsigned long long w = tile < nP ? (1ull << lim) - 1ull : ((tile - nP) == 0 ? mw0 : mw1);
          const uint32_t w_lo = (uint32_t)w, w_hi = (uint32_t)(w >> 32);
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const bool keep = ((c < 32 ? w_lo : w_hi) & (1u << (c & 31))) != 0u;
            const float v = keep ? __uint_as_float(raw[c]) : -INFINITY;
            raw[c] = __float_as_uint(v);
            mx[c & 3] = fmaxf(mx[c & 3], v);
          }
        }
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale;  // scale > 0
        const float m_new = fmaxf(m_used, tmax);
        const bool grow = m_new > m_used + kRescaleLog2;  // also true for the first finite max
        // O in TMEM holds sum_{<j} P V relative to m_used: rescale it when the
        // max grew by more than 2^8 (warp-collective TMEM access)
        if (__any_sync(0xffffffffu, grow && j > 0 && m_used > -INFINITY)) {
          if (!warp_wait(bar(B_OFULL), (uint32_t)(j - 1) & 1u, abort_flag, a.wait_cycles)) { ok_rows = false; break; }
          tc_fence_after();
          const float sc = (grow && m_used > -INFINITY) ? ex2(m_used - m_new) : 1.f;
          uint32_t ov[16];  // 16 columns at a time: with S's 64 values live, wider chunks spill registers
#pragma unroll
          for (int part = 0; part < kTcDim / 16; ++part) {
            const uint32_t oa = lane_base + kColO + 16 * part;
            tmem_ld16(oa, ov);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * sc);
            tmem_st16(oa, ov);
          }
          tmem_wait_st();
          l *= sc;
        }
        if (grow) m_used = m_new;
        const float nm = m_used == -INFINITY ? 0.f : -m_used;
        float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // P = 2^(s * scale - m) as bf16 pairs, 32 keys at a time
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(fmaf(__uint_as_float(raw[32 * h + 2 * e]), scale, nm));
            const float p1 = ex2(fmaf(__uint_as_float(raw[32 * h + 2 * e + 1]), scale, nm));
            sm4[e & 3] += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + ((j & 1) ? kColP1 : kColP0) + 16 * h, pk);
        }
        tmem_wait_st();
        l += (sm4[0] + sm4[1]) + (sm4[2] + sm4[3]);
      }
      // the last, partial prefix tile: clear the V rows past the prefix so that
      // whatever the cache holds there cannot reach P.V (0 * NaN)
      if (tile == nP - 1 && (L & (kTcKeys - 1))) {
        const int stage = j % kStages;
        if (warp_wait(bar(B_VFULL + stage), (uint32_t)(j / kStages) & 1u, abort_flag, a.wait_cycles)) {
          const int first = L & (kTcKeys - 1);
          unsigned char *vs = sm + kOffV + stage * kTileBytes;
          for (int x = r; x < (kTcKeys - first) * 16; x += 32 * kSoftmaxWarps) {
            const int row = first + (x >> 4), c = x & 15;
            *reinterpret_cast<uint4 *>(vs + (c >> 3) * kHalfBytes + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        } else {
          ok_rows = false;  // the copy may still be landing: leave the stage alone
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + (j & 1)));
      if (!__all_sync(0xffffffffu, ok_rows)) { ok_rows = false; break; }
    }
    // the last P.V must have landed before O is read
    if (ok_rows && T > 0 && !warp_wait(bar(B_OFULL), (uint32_t)(T - 1) & 1u, abort_flag, a.wait_cycles)) ok_rows = false;
  }
  __syncthreads();
  tc_fence_after();
  if (a.inputs_ready) {
    pdl_wait();     // the outputs and the workspace: the previous kernel has completed
    pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  }
  const bool aborted = *abort_flag != 0;
  if (a.S == 1) {
    // ---------------- single split: normalise and write this block's rows ----------------
    if (smx && !aborted && __any_sync(0xffffffffu, my_tok >= 0) && T > 0) {
      const uint32_t lane_base = tmem + ((uint32_t)(r & ~31) << 16);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t ov[64];
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {  // 64 columns per TMEM load, one wait each
        tmem_ld64(lane_base + kColO + 64 * h, ov);
        tmem_wait_ld();
        if (my_tok >= 0) {
          __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) +
                                (((long long)b * N + my_tok) * a.Hq + row_head[r]) * kTcDim + 64 * h;
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
            *reinterpret_cast<uint4 *>(orow + c) = v;
          }
        }
      }
      if (my_tok >= 0 && a.lse)
        a.lse[((long long)b * a.Hq + row_head[r]) * N + my_tok] =
            l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
      __syncwarp();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (aborted && t == 0) flag_status(a.dev_status, ET_DEV_TIMEOUT);
    return;
  }

  // ---------------- S splits of a tile with at most 64 real rows: merged through DSMEM ----------------
  // After one cluster barrier (every split is done with its Q, K and V
  // space), each softmax thread sends its unnormalised row straight from TMEM
  // to the shared memory of the row's owner o = row / per (slot s of o's Q/K
  // space) as fp16 scaled by the row's largest magnitude (values in [-1, 1],
  // error at most 2^-12 of that magnitude), with its (max, sum, scale); the
  // 16-byte chunk c of row r sits at c ^ (r & 15), conflict-free from one
  // thread per row and for the merge below.  A second cluster barrier (release / acquire) makes every row
  // visible to its owner, which merges its slice.  No block writes into
  // another after that barrier, so each may leave once it has merged.
  const int S = a.S;
  const int nvalid = min(kTcRows, N * a.G - mt * kTcRows);  // the real rows are a prefix of the tile
  const bool have = !aborted && T > 0;
  if (nvalid <= kDsmMaxRows) {
    const int per = (((nvalid + S - 1) / S) + 1) & ~1;  // S * per <= kDsmMaxSlots
    cluster_sync_all();  // every split is done with its Q, K and V space
    if (smx) {
      const int o = r / per, lr = r - o * per;
      float amax = 0.f;
      if (have && __any_sync(0xffffffffu, my_tok >= 0)) {
        const uint32_t lane_base = tmem + ((uint32_t)(r & ~31) << 16);
        const uint32_t dst = r < nvalid ? cl_map(sm + kOffRecv + ((size_t)s * per + lr) * kRecvRowBytes, (uint32_t)o) : 0u;
        uint32_t ov[64];
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {  // the row's largest magnitude (NaN is passed through below)
          tmem_ld64(lane_base + kColO + 64 * h, ov);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; ++c) amax = fmaxf(amax, fabsf(__uint_as_float(ov[c])));
        }
        const float inv = amax > 0.f ? 1.f / amax : 0.f;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          tmem_ld64(lane_base + kColO + 64 * h, ov);
          tmem_wait_ld();
          if (r < nvalid) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t hv[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                hv[u] = pack_f16x2(__uint_as_float(ov[8 * c + 2 * u]) * inv, __uint_as_float(ov[8 * c + 2 * u + 1]) * inv);
              asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               dst + (uint32_t)(((8 * h + c) ^ (r & 15)) << 4)),
                           "r"(hv[0]), "r"(hv[1]), "r"(hv[2]), "r"(hv[3])
                           : "memory");
            }
          }
        }
      }
      if (r < nvalid)
        cl_st_f32x4(cl_map(sm + kOffMlRecv + ((size_t)s * per + lr) * 16, (uint32_t)o), have ? m_used : -INFINITY,
                    have ? l : 0.f, amax, 0.f);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
      __syncwarp();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    cluster_sync_all();  // every split's rows and pairs have landed in their owners
    const int r0 = s * per, cnt = max(0, min(nvalid, r0 + per) - r0);
    if (!aborted && cnt > 0) {
      __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
      const float4 *mlr = reinterpret_cast<const float4 *>(sm + kOffMlRecv);
      for (int x = t; x < cnt * 32; x += kThreads) {
        const int lr = x >> 5, piece = x & 31, rr = r0 + lr;  // piece: 4 of the row's 128 values
        float M = -INFINITY;
        for (int sp = 0; sp < S; ++sp) M = fmaxf(M, mlr[sp * per + lr].x);
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < S; ++sp) {
          const float4 ml = mlr[sp * per + lr];
          if (ml.x > -INFINITY) {  // a split without keys for this row sent no row
            const float w = ex2(ml.x - M);
            Ls = fmaf(ml.y, w, Ls);
            const uint2 hp = *reinterpret_cast<const uint2 *>(sm + kOffRecv + ((size_t)sp * per + lr) * kRecvRowBytes +
                                                              (((piece >> 1) ^ (rr & 15)) << 4) + (piece & 1) * 8);
            const float ws = w * ml.z;
            const float2 p01 = __half22float2(*reinterpret_cast<const __half2 *>(&hp.x));
            const float2 p23 = __half22float2(*reinterpret_cast<const __half2 *>(&hp.y));
            acc.x = fmaf(ws, p01.x, acc.x);
            acc.y = fmaf(ws, p01.y, acc.y);
            acc.z = fmaf(ws, p23.x, acc.z);
            acc.w = fmaf(ws, p23.y, acc.w);
          }
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        uint2 v;
        v.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        v.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(O + (((long long)b * N + row_tok[rr]) * a.Hq + row_head[rr]) * kTcDim + 4 * piece) =
            v;
        if (piece == 0 && a.lse)
          a.lse[((long long)b * a.Hq + row_head[rr]) * N + row_tok[rr]] =
              Ls > 0.f ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
      }
    }
    if (aborted && t == 0) flag_status(a.dev_status, ET_DEV_TIMEOUT);
    return;
  }

  // ---------------- S splits, larger tiles: partial rows through L2, merged by their owners ----------------
  // Each split writes the unnormalised fp32 rows of its real tokens straight
  // from TMEM to the workspace (one 512-byte row per softmax thread) and
  // posts (max, sum) per row.  The S splits of a tile form one cluster: after
  // one cluster barrier, split s merges rows [s * per, (s + 1) * per) of the
  // tile from all S partials (the pairs and the rows are loaded in one round),
  // then drops those scratch lines from L2 so that they are never written
  // back to DRAM.
  const long long tile_id = (long long)blockIdx.z * gridDim.y + blockIdx.y;
  const long long n_tiles = (long long)gridDim.y * gridDim.z;
  float *ws_o = a.ws;                                                                  // [tiles][S][128][128]
  float2 *ws_ml = reinterpret_cast<float2 *>(a.ws + n_tiles * S * kTcRows * kTcDim);  // [tiles][S][128]
  if (smx) {
    if (have && __any_sync(0xffffffffu, my_tok >= 0)) {
      const uint32_t lane_base = tmem + ((uint32_t)(r & ~31) << 16);
      float4 *dst = reinterpret_cast<float4 *>(ws_o + ((tile_id * S + s) * kTcRows + r) * kTcDim);
      uint32_t ov[64];
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {  // 64 columns per TMEM load, one wait each
        tmem_ld64(lane_base + kColO + 64 * h, ov);
        tmem_wait_ld();
        if (my_tok >= 0) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            dst[16 * h + c] = make_float4(__uint_as_float(ov[4 * c]), __uint_as_float(ov[4 * c + 1]),
                                          __uint_as_float(ov[4 * c + 2]), __uint_as_float(ov[4 * c + 3]));
        }
      }
    }
    if (r < nvalid) ws_ml[(tile_id * S + s) * kTcRows + r] = make_float2(have ? m_used : -INFINITY, have ? l : 0.f);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  cluster_sync_all();  // release / acquire at cluster scope: every split's rows are in L2
  if (aborted) {
    if (t == 0) flag_status(a.dev_status, ET_DEV_TIMEOUT);
    return;
  }
  const int per = (nvalid + S - 1) / S;  // the real rows, spread over every split
  const int r0 = s * per, r1 = min(nvalid, r0 + per);
  if (r1 <= r0) return;
  __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
  const float4 *src = reinterpret_cast<const float4 *>(ws_o + tile_id * S * (kTcRows * kTcDim));
  const float2 *mlt = ws_ml + tile_id * S * kTcRows;
  for (int x = t; x < (r1 - r0) * 32; x += kThreads) {
    const int rr = r0 + (x >> 5), chunk = x & 31;
    float2 ml[kTcMaxSplits];
    float4 p[kTcMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kTcMaxSplits; ++sp) {  // every load in flight before any arithmetic
      ml[sp] = sp < S ? __ldcg(mlt + sp * kTcRows + rr) : make_float2(-INFINITY, 0.f);
      p[sp] = sp < S ? __ldcg(src + (sp * kTcRows + rr) * 32 + chunk) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kTcMaxSplits; ++sp) M = fmaxf(M, ml[sp].x);
    float Ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < kTcMaxSplits; ++sp) {
      if (ml[sp].x > -INFINITY) {  // a split without keys for this row wrote no partial row
        const float w = exp2f(ml[sp].x - M);
        Ls = fmaf(ml[sp].y, w, Ls);
        acc.x = fmaf(w, p[sp].x, acc.x);
        acc.y = fmaf(w, p[sp].y, acc.y);
        acc.z = fmaf(w, p[sp].z, acc.z);
        acc.w = fmaf(w, p[sp].w, acc.w);
      }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    uint2 v;
    v.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    v.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(O + (((long long)b * N + row_tok[rr]) * a.Hq + row_head[rr]) * kTcDim + 4 * chunk) = v;
    if (chunk == 0 && a.lse)
      a.lse[((long long)b * a.Hq + row_head[rr]) * N + row_tok[rr]] =
          Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();  // every read of this block's rows has returned
  for (int x = t; x < (r1 - r0) * S * 4; x += kThreads) {
    const int line = x & 3, lr = (x >> 2) % (r1 - r0), sp = (x >> 2) / (r1 - r0);
    discard_l2_line(src + (sp * kTcRows + r0 + lr) * 32 + line * 8);
  }
}

// ---------------------------------------------------------------------------
// host: tensor maps and launch
// ---------------------------------------------------------------------------
bool make_map_2d(CUtensorMap *m, const void *base, long long rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)kTcDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kTcDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTcKeys};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tree K/V [B*N rows][Hkv][d]: box = 64 rows of one head
bool make_map_tree(CUtensorMap *m, const void *base, int Hkv, long long rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)kTcDim, (cuuint64_t)Hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kTcDim * 2, (cuuint64_t)Hkv * kTcDim * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcKeys};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [B*N tokens][Hkv][G][d]: box = 128/G tokens x G heads of one KV head,
// rows ordered (token, head in group) like the tile
bool make_map_q(CUtensorMap *m, const void *base, int G, int Hkv, long long tokens) {
  const cuuint64_t dims[4] = {(cuuint64_t)kTcDim, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)tokens};
  const cuuint64_t strides[3] = {(cuuint64_t)kTcDim * 2, (cuuint64_t)G * kTcDim * 2,
                                 (cuuint64_t)Hkv * G * kTcDim * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(kTcRows / G)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr() {
  const cudaError_t e = et_smem_attr((const void *)k_attn_tc<false>, (int)kSmemBytes);
  return e != cudaSuccess ? e : et_smem_attr((const void *)k_attn_tc<true>, (int)kSmemBytes);
}

// clusters of more than 8 blocks (the portable limit) need an opt-in per
// device; thread-safe
cudaError_t allow_big_clusters() {
  static std::mutex mu;
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute((const void *)k_attn_tc<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void *)k_attn_tc<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[dev] = 1;
  return e;
}

}  // namespace

et_status tc_attention_launch(const TcLaunch &a, cudaStream_t stream) {
  if (!encode_fn()) return ET_ERR_CUDA;
  if (a.S < 1 || a.S > kTcMaxSplits) return ET_ERR_UNSUPPORTED;
  if (a.kv_rows >= (1ll << 31) || (long long)a.B * a.N >= (1ll << 31)) return ET_ERR_UNSUPPORTED;
  if (a.S > 1 && !a.ws) return ET_ERR_WORKSPACE;
  CUtensorMap m_kp, m_vp, m_kt, m_vt, m_q;
  const long long tree_rows = (long long)a.B * a.N;
  bool ok = make_map_tree(&m_kt, a.kt, a.Hkv, tree_rows) && make_map_tree(&m_vt, a.vt, a.Hkv, tree_rows);
  if (a.kp && a.vp && a.kv_rows > 0) {
    ok = ok && make_map_2d(&m_kp, a.kp, a.kv_rows) && make_map_2d(&m_vp, a.vp, a.kv_rows);
  } else {  // no prefix anywhere: a valid map the kernel never uses
    ok = ok && make_map_2d(&m_kp, a.kt, tree_rows * a.Hkv) && make_map_2d(&m_vp, a.vt, tree_rows * a.Hkv);
  }
  TcLaunch la = a;
  la.q_tma = (a.G <= kTcRows && kTcRows % a.G == 0) ? 1 : 0;
  la.wait_cycles = et_wait_limit_cycles();
  if (la.q_tma) ok = ok && make_map_q(&m_q, a.q, a.G, a.Hkv, tree_rows);
  else m_q = m_kt;  // not read
  if (!ok) return ET_ERR_INVALID_ARG;
  if (set_smem_attr() != cudaSuccess) return ET_ERR_CUDA;
  if (a.S > 8 && allow_big_clusters() != cudaSuccess) return ET_ERR_CUDA;
  if (a.B > 1 && a.B <= kLptMaxB)
    return et_launch(k_attn_tc<true>, dim3(a.S, a.Hkv * a.MT, a.B), dim3(kThreads), kSmemBytes, stream,
                     a.S > 1 ? a.S : 0, m_kp, m_vp, m_kt, m_vt, m_q, la);
  return et_launch(k_attn_tc<false>, dim3(a.S, a.Hkv * a.MT, a.B), dim3(kThreads), kSmemBytes, stream,
                   a.S > 1 ? a.S : 0, m_kp, m_vp, m_kt, m_vt, m_q, la);
}

}  // namespace et
