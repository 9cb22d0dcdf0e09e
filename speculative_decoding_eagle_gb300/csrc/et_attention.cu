// Tree-masked attention on sm_103a (EAGLE-2 article on sbmmt.com, attention
// mask paragraph: every flattened draft token attends to the KV prefix and
// to its own in-tree ancestors only).
//
// Paths:
//  * fp32: CUDA-core kernel, one block per (row, head, sequence);
//  * bf16, legacy tensor cores (mma.sync m16n8k16): split-KV blocks over
//    (split, KV head x row tile, sequence); a row tile holds 64 (token,
//    query head) rows of one KV head, so GQA groups share every K/V tile;
//    K/V stream through a cp.async double buffer with an XOR-swizzled
//    layout; splits are merged by the last block to finish (no waits);
//  * bf16 with d = 128: the tcgen05 / TMA / TMEM kernel of et_attention_tc.cu
//    (the default; the mma.sync kernel stays selectable and covers d = 64).
#include <cuda_bf16.h>

#include <atomic>

#include "et_attn_internal.h"
#include "et_common.cuh"

namespace et {

// ---------------------------------------------------------------------------
// common: where row r of a (b, g, row tile) lives
// ---------------------------------------------------------------------------
struct AttnArgs {
  int B, N, Hq, Hkv, G, d, MT, S;   // MT row tiles per KV head, S splits
  float scale_log2;                 // scale * log2(e)
  int W;                            // mask words per row
  const void *q, *kp, *vp, *kt, *vt;
  const long long *kv_row0;
  const int *prefix_len;
  long long kv_rows, kv_head_stride;
  const unsigned long long *mask;
  void *out;
  float *lse;
  int *dev_status;
  float *part_o;            // [tiles][S][64][d] fp32 (unnormalised)
  float2 *part_ml;          // [tiles][S][64] (max in log2 units, sum)
  unsigned int *cnt;        // [tiles]
};

// ---------------------------------------------------------------------------
// fp32 CUDA-core path
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) k_attn_f32(AttnArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  constexpr int PL = D / 32;  // dims per lane
  __shared__ float qs[D];
  __shared__ float wm[4], wl[4];
  __shared__ float wacc[4][D];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / a.G;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const float *q = static_cast<const float *>(a.q) + (((long long)b * a.N + i) * a.Hq + h) * D;
  for (int c = t; c < D; c += 128) qs[c] = q[c];
  __syncthreads();
  const int L = a.prefix_len[b];
  const long long S_b = a.kv_head_stride > 0 ? a.kv_head_stride : L;
  const long long row0 = a.kv_row0 ? a.kv_row0[b] : 0;
  const unsigned long long *mrow = a.mask + ((long long)b * a.N + i) * a.W;
  float m = -INFINITY, l = 0.f, acc[PL];
#pragma unroll
  for (int c = 0; c < PL; ++c) acc[c] = 0.f;
  int bad = 0;
  for (int j = warp; j < L + a.N; j += 4) {
    const float *kr, *vr;
    if (j < L) {
      const long long r = row0 + g * S_b + j;
      if (r < 0 || r >= a.kv_rows) { bad = 1; continue; }
      kr = static_cast<const float *>(a.kp) + r * D;
      vr = static_cast<const float *>(a.vp) + r * D;
    } else {
      const int tt = j - L;
      if (!((mrow[tt >> 6] >> (tt & 63)) & 1ull)) continue;
      kr = static_cast<const float *>(a.kt) + (((long long)b * a.N + tt) * a.Hkv + g) * D;
      vr = static_cast<const float *>(a.vt) + (((long long)b * a.N + tt) * a.Hkv + g) * D;
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < PL; ++c) s = fmaf(qs[lane + 32 * c], kr[lane + 32 * c], s);
    s = warp_sum(s) * a.scale_log2;
    const float mn = fmaxf(m, s);
    const float corr = exp2f(m - mn);
    const float p = exp2f(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int c = 0; c < PL; ++c) acc[c] = fmaf(p, vr[lane + 32 * c], acc[c] * corr);
    m = mn;
  }
  if (lane == 0) { wm[warp] = m; wl[warp] = l; }
#pragma unroll
  for (int c = 0; c < PL; ++c) wacc[warp][lane + 32 * c] = acc[c];
  __syncthreads();
  float M = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
  float Ls = 0.f, wts[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wts[w] = wm[w] > -INFINITY ? exp2f(wm[w] - M) : 0.f;
    Ls += wl[w] * wts[w];
  }
  float *o = static_cast<float *>(a.out) + (((long long)b * a.N + i) * a.Hq + h) * D;
  for (int c = t; c < D; c += 128) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) v += wacc[w][c] * wts[w];
    o[c] = Ls > 0.f ? v / Ls : 0.f;
  }
  if (t == 0 && a.lse) a.lse[((long long)b * a.Hq + h) * a.N + i] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
  if (bad) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
}

// ---------------------------------------------------------------------------
// bf16 path on mma.sync (m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------
constexpr int kMmaThreads = 128;   // 4 warps x 16 rows
constexpr int kRows = 64;          // rows per tile
constexpr int kKeys = 64;          // keys per KV tile

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 bytes read -> 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int n>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(n)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// byte offset of 16-byte chunk `c` of row `r` in a [rows][D] bf16 tile whose
// chunks are XOR-swizzled by the row (conflict-free ldmatrix)
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Work of one block: tiles [t0, t1) of the sequence's virtual key list
// (prefix tiles, then ceil(N/64) tree tiles).
__device__ __forceinline__ void split_range(int L, int N, int S, int s, int &t0, int &t1, int &nP) {
  nP = (L + kKeys - 1) / kKeys;
  const int T = nP + (N + kKeys - 1) / kKeys;
  const int per = (T + S - 1) / S;
  t0 = s * per;
  t1 = min(T, t0 + per);
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads, 2) k_attn_mma(AttnArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char *qs = sm;                            // [64][D]
  unsigned char *ks = sm + kRows * D * 2;            // [2][64][D]
  unsigned char *vs = ks + 2 * kKeys * D * 2;        // [2][64][D]
  __shared__ int sflag;
  __shared__ int row_tok[kRows], row_head[kRows];

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int s = blockIdx.x;
  const int g = blockIdx.y / a.MT, mt = blockIdx.y - g * a.MT;
  const int b = blockIdx.z;
  const int N = a.N;
  const int L = a.prefix_len[b];
  const long long S_b = a.kv_head_stride > 0 ? a.kv_head_stride : L;
  const long long row0 = a.kv_row0 ? a.kv_row0[b] : 0;
  const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *KP = static_cast<const __nv_bfloat16 *>(a.kp);
  const __nv_bfloat16 *VP = static_cast<const __nv_bfloat16 *>(a.vp);
  const __nv_bfloat16 *KT = static_cast<const __nv_bfloat16 *>(a.kt);
  const __nv_bfloat16 *VT = static_cast<const __nv_bfloat16 *>(a.vt);
  int bad = 0;

  if (t < kRows) {
    const int R = mt * kRows + t;
    const int i = R / a.G;
    row_tok[t] = i < N ? i : -1;
    row_head[t] = g * a.G + (R - i * a.G);
  }
  __syncthreads();
  // Q tile -> smem (invalid rows are zero)
  for (int x = t; x < kRows * CH; x += kMmaThreads) {
    const int r = x / CH, c = x - r * CH;
    const int i = row_tok[r];
    const __nv_bfloat16 *src = Q + (((long long)b * N + (i < 0 ? 0 : i)) * a.Hq + row_head[r]) * D + c * 8;
    cp_async16(smem_u32(qs + swz<D>(r, c)), src, i >= 0);
  }
  cp_async_commit();

  int t0, t1, nP;
  split_range(L, N, a.S, s, t0, t1, nP);

  auto load_tile = [&](int tile, int stage) {
    unsigned char *kd = ks + stage * kKeys * D * 2;
    unsigned char *vd = vs + stage * kKeys * D * 2;
    for (int x = t; x < kKeys * CH; x += kMmaThreads) {
      const int r = x / CH, c = x - r * CH;
      const __nv_bfloat16 *ksrc = KT, *vsrc = VT;  // a valid address even for zero-byte copies
      bool valid;
      if (tile < nP) {
        const int j = tile * kKeys + r;
        const long long row = row0 + g * S_b + j;
        valid = j < L;
        if (valid && (row < 0 || row >= a.kv_rows)) { valid = false; bad = 1; }
        if (valid) { ksrc = KP + row * D + c * 8; vsrc = VP + row * D + c * 8; }
      } else {
        const int tt = (tile - nP) * kKeys + r;
        valid = tt < N;
        if (valid) {
          const long long off = (((long long)b * N + tt) * a.Hkv + g) * D + c * 8;
          ksrc = KT + off;
          vsrc = VT + off;
        }
      }
      cp_async16(smem_u32(kd + swz<D>(r, c)), ksrc, valid);
      cp_async16(smem_u32(vd + swz<D>(r, c)), vsrc, valid);
    }
  };

  // per-thread rows: g8 = lane>>2 and g8+8 within the warp's 16
  const int tq = lane & 3, g8 = lane >> 2;
  const int r0 = warp * 16 + g8, r1 = r0 + 8;
  float m_[2] = {-INFINITY, -INFINITY}, l_[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  unsigned long long mk[2][2] = {{0ull, 0ull}, {0ull, 0ull}};
  {
    const int i0 = row_tok[r0], i1 = row_tok[r1];
    for (int w = 0; w < a.W; ++w) {
      if (i0 >= 0) mk[0][w] = a.mask[((long long)b * N + i0) * a.W + w];
      if (i1 >= 0) mk[1][w] = a.mask[((long long)b * N + i1) * a.W + w];
    }
  }
  uint32_t qf[D / 16][4];
  bool qloaded = false;

  if (t0 < t1) load_tile(t0, 0);
  cp_async_commit();
  for (int tile = t0; tile < t1; ++tile) {
    const int stage = (tile - t0) & 1;
    if (tile + 1 < t1) load_tile(tile + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (!qloaded) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_u32(qs + swz<D>(warp * 16 + (lane & 15), 2 * kk + (lane >> 4))), qf[kk][0], qf[kk][1],
                qf[kk][2], qf[kk][3]);
      qloaded = true;
    }
    const unsigned char *kd = ks + stage * kKeys * D * 2;
    const unsigned char *vd = vs + stage * kKeys * D * 2;
    // S = Q K^T for 64 keys
    float sc[kKeys / 8][4];
#pragma unroll
    for (int j = 0; j < kKeys / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < kKeys / 8; ++j) {
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(kd + swz<D>(8 * j + (lane & 7), 2 * kk + (lane >> 3))), b0, b1, b2, b3);
        mma_bf16(sc[j], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(sc[j], qf[kk + 1][0], qf[kk + 1][1], qf[kk + 1][2], qf[kk + 1][3], b2, b3);
      }
    }
    // mask + online softmax (log2 domain)
    const bool is_tree = tile >= nP;
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < kKeys / 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = 8 * j + 2 * tq + (e & 1);
        const int rr = e >> 1;
        bool ok;
        if (!is_tree) {
          ok = tile * kKeys + n < L;
        } else {
          const int tt = (tile - nP) * kKeys + n;
          ok = tt < N && ((mk[rr][tt >> 6] >> (tt & 63)) & 1ull);
        }
        const float v = ok ? sc[j][e] * a.scale_log2 : -INFINITY;
        sc[j][e] = v;
        tmax[rr] = fmaxf(tmax[rr], v);
      }
    }
    float corr[2], msafe[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 1));
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 2));
      const float mn = fmaxf(m_[rr], tmax[rr]);
      msafe[rr] = mn == -INFINITY ? 0.f : mn;
      corr[rr] = exp2f(m_[rr] - msafe[rr]);
      m_[rr] = mn;
      l_[rr] *= corr[rr];
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      o[j][0] *= corr[0]; o[j][1] *= corr[0];
      o[j][2] *= corr[1]; o[j][3] *= corr[1];
    }
    uint32_t pa[kKeys / 16][4];
#pragma unroll
    for (int j = 0; j < kKeys / 8; ++j) {
      const float p0 = exp2f(sc[j][0] - msafe[0]), p1 = exp2f(sc[j][1] - msafe[0]);
      const float p2 = exp2f(sc[j][2] - msafe[1]), p3 = exp2f(sc[j][3] - msafe[1]);
      l_[0] += p0 + p1;
      l_[1] += p2 + p3;
      pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < kKeys / 16; ++kk) {
#pragma unroll
      for (int j = 0; j < D / 8; j += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(vd + swz<D>(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), j + (lane >> 4))), b0, b1,
                  b2, b3);
        mma_bf16(o[j], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma_bf16(o[j + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // quad-reduce the row sums
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 1);
    l_[rr] += __shfl_xor_sync(0xffffffffu, l_[rr], 2);
  }
  if (bad) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  const long long tile_id = ((long long)b * a.Hkv + g) * a.MT + mt;
  if (a.S == 1) {
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = rr ? r1 : r0;
      const int i = row_tok[r];
      if (i < 0) continue;
      const float inv = l_[rr] > 0.f ? 1.f / l_[rr] : 0.f;
      __nv_bfloat16 *orow = O + (((long long)b * N + i) * a.Hq + row_head[r]) * D;
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        *reinterpret_cast<__nv_bfloat162 *>(orow + 8 * j + 2 * tq) =
            __floats2bfloat162_rn(o[j][2 * rr] * inv, o[j][2 * rr + 1] * inv);
      if (a.lse && tq == 0)
        a.lse[((long long)b * a.Hq + row_head[r]) * N + i] =
            l_[rr] > 0.f ? (m_[rr] + log2f(l_[rr])) * 0.69314718055994531f : -INFINITY;
    }
    return;
  }
  // ---- split partials, then the last block of this tile merges them ----
  float *po = a.part_o + ((tile_id * a.S + s) * kRows) * D;
  float2 *pml = a.part_ml + (tile_id * a.S + s) * kRows;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rr ? r1 : r0;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
      *reinterpret_cast<float2 *>(po + r * D + 8 * j + 2 * tq) = make_float2(o[j][2 * rr], o[j][2 * rr + 1]);
    if (tq == 0) pml[r] = make_float2(m_[rr], l_[rr]);
  }
  if (!arrive_last(&a.cnt[tile_id], (unsigned)a.S, &sflag)) return;

  float *wts = reinterpret_cast<float *>(ks);  // [64][S] merge weights (reuses the K buffers)
  float *lsum = reinterpret_cast<float *>(vs);  // [64]
  if (t < kRows) {
    const float2 *ml = a.part_ml + tile_id * a.S * kRows;
    float M = -INFINITY;
    for (int x = 0; x < a.S; ++x) M = fmaxf(M, ld_cg(&ml[x * kRows + t].x));
    float Ls = 0.f;
    for (int x = 0; x < a.S; ++x) {
      const float2 v = __ldcg(&ml[x * kRows + t]);
      const float w = v.x > -INFINITY ? exp2f(v.x - M) : 0.f;
      wts[t * a.S + x] = w;
      Ls += v.y * w;
    }
    lsum[t] = Ls;
    const int i = row_tok[t];
    if (i >= 0 && a.lse)
      a.lse[((long long)b * a.Hq + row_head[t]) * N + i] = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  const float *pall = a.part_o + tile_id * a.S * kRows * D;
  __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
  for (int x = t; x < kRows * (D / 2); x += kMmaThreads) {
    const int r = x / (D / 2), c = 2 * (x - r * (D / 2));
    const int i = row_tok[r];
    if (i < 0) continue;
    float v0 = 0.f, v1 = 0.f;
    for (int sp = 0; sp < a.S; ++sp) {
      const float w = wts[r * a.S + sp];
      if (w == 0.f) continue;
      const float2 p = __ldcg(reinterpret_cast<const float2 *>(pall + ((long long)sp * kRows + r) * D + c));
      v0 = fmaf(w, p.x, v0);
      v1 = fmaf(w, p.y, v1);
    }
    const float inv = lsum[r] > 0.f ? 1.f / lsum[r] : 0.f;
    *reinterpret_cast<__nv_bfloat162 *>(O + (((long long)b * N + i) * a.Hq + row_head[r]) * D + c) =
        __floats2bfloat162_rn(v0 * inv, v1 * inv);
  }
}

}  // namespace et

using namespace et;

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int sm_count() {
  static std::atomic<int> cached[64];  // zero-initialised (static storage)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) cudaGetLastError();
  if (dev < 0 || dev >= 64) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cudaGetLastError();
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static bool attn_shape_ok(const et_attn_shape *s) {
  if (!s) return false;
  if (s->B < 1 || s->N < 1 || s->N > kMaxN || s->Hq < 1 || s->Hkv < 1 || s->Hq % s->Hkv) return false;
  if (s->d != 64 && s->d != 128) return false;
  if (s->dtype != ET_BF16 && s->dtype != ET_F32) return false;
  if (s->max_prefix < 0 || s->kv_rows < 0 || s->kv_head_stride < 0 || s->num_splits < 0) return false;
  if (s->impl < 0 || s->impl > 2) return false;
  if (s->flags & ~ET_ATTN_INPUTS_READY) return false;
  if (!(s->scale > 0.f)) return false;
  return true;
}

// How one call is carried out: path, row-tile height, tiles and splits.
struct AttnPlan {
  int impl;   // 0 fp32 CUDA cores, 1 mma.sync, 2 tcgen05
  int rows;   // rows per tile
  int MT;     // row tiles per KV head
  int S;      // KV splits
  size_t ws;  // workspace bytes
  size_t cnt_off, ml_off, po_off;
};

static bool make_plan(const et_attn_shape *s, AttnPlan *p) {
  if (!attn_shape_ok(s)) return false;
  const bool tc_ok = s->dtype == ET_BF16 && s->d == kTcDim;
  if (s->dtype == ET_F32) {
    if (s->impl != 0) return false;
    p->impl = 0; p->rows = 1; p->MT = s->N; p->S = 1;
  } else if (s->impl == 2 || (s->impl == 0 && tc_ok)) {
    if (!tc_ok) return false;
    p->impl = 2; p->rows = kTcRows;
  } else {
    p->impl = 1; p->rows = kRows;
  }
  const int G = s->Hq / s->Hkv;
  const int T = (s->max_prefix + kKeys - 1) / kKeys + (s->N + kKeys - 1) / kKeys;
  if (p->impl != 0) {
    p->MT = (s->N * G + p->rows - 1) / p->rows;
    const long long base = (long long)s->B * s->Hkv * p->MT;
    const int cap = T / 2 > 0 ? T / 2 : 1;  // at least two K/V tiles per split
    int S = s->num_splits;
    if (p->impl == 2) {
      // the splits of a row tile form one thread-block cluster (<= 8 blocks);
      // two blocks fit per SM: aim at ~1.7 blocks per SM so that the
      // clusters still find room in one wave (measured on GB300: 6 splits for
      // 40 heads and 5 for 48 row tiles beat both fewer and more), and at
      // about 3 K/V tiles per split: below that the split merge outweighs
      // the shorter loop (7B heads, prefix 1024, 17 tiles: 10.45 us at 6
      // splits, 10.8 at 4 and 5, 11.6 at 3)
      if (S <= 0) {
        S = (int)((17LL * sm_count()) / (10LL * base));
        // a ragged batch whose blocks go out longest prefix first
        // (kLptMaxB) runs in several waves: about five blocks per SM keep
        // the last wave short (7B heads, prefixes 512..16384, measured on
        // GB300: 4 sequences best at 4 splits, 8 at 2-4, 16 at 2, 32 at 1)
        if (s->B > 1 && s->B <= kLptMaxB) {
          const int waves = (int)((5LL * sm_count() + base - 1) / base);
          if (S < waves) S = waves;
        }
        const int by_tiles = (T + 2) / 3;  // ceil(T / 3)
        if (S > by_tiles) S = by_tiles;
        if (S > cap) S = cap;
        if (S > 8) S = 8;  // the portable cluster size (larger clusters are an explicit choice)
        if (S < 1) S = 1;
      }
      if (S > kTcMaxSplits) S = kTcMaxSplits;
    } else if (S <= 0) {  // two resident blocks per SM
      S = (int)((2LL * sm_count() + base - 1) / base);
      if (S > cap) S = cap;
    }
    if (S > T) S = T;
    if (S > 32) S = 32;
    if (S < 1) S = 1;
    p->S = S;
  }
  p->ws = 0;
  p->cnt_off = p->ml_off = p->po_off = 0;
  if (p->impl == 2) p->ws = tc_workspace_bytes((long long)s->B * s->Hkv * p->MT, p->S);
  if (p->impl == 1 && p->S > 1) {
    const size_t tiles = (size_t)s->B * s->Hkv * p->MT;
    const size_t cnt = (tiles * sizeof(unsigned int) + 255) & ~(size_t)255;
    const size_t ml = (tiles * p->S * p->rows * sizeof(float2) + 255) & ~(size_t)255;
    p->cnt_off = 0;
    p->ml_off = cnt;
    p->po_off = cnt + ml;
    p->ws = cnt + ml + tiles * p->S * p->rows * (size_t)s->d * sizeof(float);
  }
  return true;
}

extern "C" int32_t et_tree_attention_splits(const et_attn_shape *s) {
  AttnPlan p;
  return make_plan(s, &p) ? p.S : -1;
}

extern "C" size_t et_tree_attention_workspace_size(const et_attn_shape *s) {
  AttnPlan p;
  return make_plan(s, &p) ? p.ws : 0;
}

extern "C" et_status et_tree_attention(const et_attn_shape *shape, const void *q, const void *k_prefix,
                                       const void *v_prefix, const int64_t *kv_row0, const int32_t *prefix_len,
                                       const void *k_tree, const void *v_tree, const uint64_t *mask, void *out,
                                       float *lse, int32_t *dev_status, void *ws, size_t ws_bytes,
                                       et_stream_t stream) {
  ET_RETURN_IF(!shape, ET_ERR_INVALID_ARG);
  if (shape->d != 64 && shape->d != 128 && shape->d > 0) return ET_ERR_UNSUPPORTED;
  ET_RETURN_IF(!attn_shape_ok(shape), ET_ERR_INVALID_ARG);
  AttnPlan plan;
  if (!make_plan(shape, &plan)) return ET_ERR_UNSUPPORTED;
  ET_RETURN_IF(!q || !k_tree || !v_tree || !mask || !out || !prefix_len, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(shape->max_prefix > 0 && (!k_prefix || !v_prefix || !kv_row0), ET_ERR_INVALID_ARG);
  const size_t al = shape->dtype == ET_BF16 ? 16 : 4;
  ET_RETURN_IF(!et_aligned(q, al) || !et_aligned(k_tree, al) || !et_aligned(v_tree, al) || !et_aligned(out, al) ||
                   (k_prefix && !et_aligned(k_prefix, al)) || (v_prefix && !et_aligned(v_prefix, al)) ||
                   !et_aligned(mask, 8),
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(plan.ws > 0 && (!ws || ws_bytes < plan.ws || !et_aligned(ws, 256)), ET_ERR_WORKSPACE);
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char *wsb = static_cast<unsigned char *>(ws);

  if (plan.impl == 2) {
    TcLaunch t{};
    t.B = shape->B; t.N = shape->N; t.Hq = shape->Hq; t.Hkv = shape->Hkv; t.G = shape->Hq / shape->Hkv;
    t.MT = plan.MT; t.S = plan.S; t.W = (shape->N + 63) / 64;
    t.inputs_ready = (shape->flags & ET_ATTN_INPUTS_READY) ? 1 : 0;
    t.scale_log2 = shape->scale * 1.4426950408889634f;
    t.q = q; t.kp = k_prefix; t.vp = v_prefix; t.kt = k_tree; t.vt = v_tree;
    t.kv_row0 = reinterpret_cast<const long long *>(kv_row0);
    t.prefix_len = prefix_len;
    t.kv_rows = shape->kv_rows;
    t.kv_head_stride = shape->kv_head_stride;
    t.mask = reinterpret_cast<const unsigned long long *>(mask);
    t.out = out; t.lse = lse; t.dev_status = dev_status;
    t.ws = static_cast<float *>(ws);
    ET_RETURN_IF((long long)t.Hkv * t.MT > 65535 || t.B > 65535, ET_ERR_UNSUPPORTED);
    return tc_attention_launch(t, st);
  }

  AttnArgs a{};
  a.B = shape->B; a.N = shape->N; a.Hq = shape->Hq; a.Hkv = shape->Hkv; a.G = shape->Hq / shape->Hkv;
  a.d = shape->d; a.MT = plan.MT; a.S = plan.S;
  a.scale_log2 = shape->scale * 1.4426950408889634f;
  a.W = (shape->N + 63) / 64;
  a.q = q; a.kp = k_prefix; a.vp = v_prefix; a.kt = k_tree; a.vt = v_tree;
  a.kv_row0 = reinterpret_cast<const long long *>(kv_row0);
  a.prefix_len = prefix_len;
  a.kv_rows = shape->kv_rows;
  a.kv_head_stride = shape->kv_head_stride;
  a.mask = reinterpret_cast<const unsigned long long *>(mask);
  a.out = out; a.lse = lse; a.dev_status = dev_status;
  if (plan.impl == 0) {
    dim3 grid(shape->N, shape->Hq, shape->B);
    if (shape->d == 64) return et_launch(k_attn_f32<64>, grid, dim3(128), 0, st, 0, a);
    return et_launch(k_attn_f32<128>, grid, dim3(128), 0, st, 0, a);
  }
  if (a.S > 1) {
    a.cnt = reinterpret_cast<unsigned int *>(wsb + plan.cnt_off);
    a.part_ml = reinterpret_cast<float2 *>(wsb + plan.ml_off);
    a.part_o = reinterpret_cast<float *>(wsb + plan.po_off);
  }
  ET_RETURN_IF((long long)a.Hkv * a.MT > 65535 || a.B > 65535, ET_ERR_UNSUPPORTED);
  dim3 grid(a.S, a.Hkv * a.MT, a.B);
  if (shape->d == 64) {
    const int smem = kRows * 64 * 2 + 4 * kKeys * 64 * 2;
    ET_RETURN_IF(et_smem_attr((const void *)k_attn_mma<64>, smem) != cudaSuccess, ET_ERR_CUDA);
    return et_launch(k_attn_mma<64>, grid, dim3(kMmaThreads), smem, st, 0, a);
  } else {
    const int smem = kRows * 128 * 2 + 4 * kKeys * 128 * 2;
    ET_RETURN_IF(et_smem_attr((const void *)k_attn_mma<128>, smem) != cudaSuccess, ET_ERR_CUDA);
    return et_launch(k_attn_mma<128>, grid, dim3(kMmaThreads), smem, st, 0, a);
  }
}
