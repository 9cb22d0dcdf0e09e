// Dynamic draft tree on sm_103a: expansion (log-softmax + top-k + path value
// + top-m frontier), rerank (top-n + flatten) and the ancestor mask /
// position ids.  Follows the EAGLE-2 article on sbmmt.com ("Up to 5x lossless
// acceleration: EAGLE-2 lets an RTX 3060 generate faster than an A100"):
// expansion phase, reranking phase, attention-mask example and the
// position-encoding sentence.
#include <atomic>

#include "et_common.cuh"

namespace et {

// ---------------------------------------------------------------------------
// expand
// ---------------------------------------------------------------------------
constexpr int kExpThreads = 256;
constexpr int kExpVec = 2;                               // float4 loads per thread
constexpr int kExpChunk = kExpThreads * 4 * kExpVec;     // logits per block

struct ExpandArgs {
  const float *logits;
  long long row_stride;
  const int32_t *row_of_node;
  int vec4;
  int B, V, k, m, C, layer, m_l, base_next, m_next, nchunk;
  et_tree tree;
  int32_t *dev_status;
  float *part;             // [B*m_l][nchunk][2 + 2k]
  unsigned int *row_cnt;   // [B*m_l]
  unsigned int *seq_cnt;   // [B]
};

// Loads this block's slice of a logit row (128-bit loads when aligned);
// out-of-row slots get -inf with id INT_MAX so they rank after every token.
template <int NV>
__device__ __forceinline__ void load_chunk(const float *zrow, int V, int c0, int vec4, float (&v)[4 * NV],
                                           int &flag) {
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int e0 = c0 + (u * kExpThreads + threadIdx.x) * 4;
    if (zrow && vec4 && e0 + 3 < V) {
      float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u + 0] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < V) ? __ldcs(zrow + e0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (e0 + j < V) v[4 * u + j] = sanitize_logit(v[4 * u + j], flag);
  }
}

__device__ __forceinline__ int chunk_id(int c0, int j, int V) {
  const int e = c0 + ((j >> 2) * kExpThreads + threadIdx.x) * 4 + (j & 3);
  return e < V ? e : 0x7fffffff;
}

__global__ void __launch_bounds__(kExpThreads) k_expand(ExpandArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  extern __shared__ unsigned char smem_raw[];
  float *mz = reinterpret_cast<float *>(smem_raw);              // [nchunk*k]
  int *mi = reinterpret_cast<int *>(mz + a.nchunk * a.k);       // [nchunk*k]
  __shared__ float redz[32];
  __shared__ int redi[32];
  __shared__ float wz[kExpThreads / 32][kMaxTopk];
  __shared__ int wi[kExpThreads / 32][kMaxTopk];
  __shared__ float topz[kMaxTopk];
  __shared__ int topi[kMaxTopk];
  __shared__ unsigned long long red64[32];
  __shared__ int sel[kMaxM];
  __shared__ int sflag;

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int row = blockIdx.y, c = blockIdx.x;
  const int b = row / a.m_l, s = row - b * a.m_l;
  const int k = a.k;
  int flag = 0, bad = 0;

  int node = -1;
  if (a.layer > 0) {
    node = a.tree.frontier[b * a.m + s];
    if (node < 0 || node >= a.C) bad = 1;
  }
  const float *zrow = nullptr;
  if (!bad) {
    long long r = a.row_of_node ? (long long)a.row_of_node[(long long)b * (a.C + 1) + node + 1] : (long long)row;
    if (r < 0) bad = 1;
    else zrow = a.logits + r * a.row_stride;
  }

  float v[4 * kExpVec];
  const int c0 = c * kExpChunk;
  load_chunk<kExpVec>(zrow, a.V, c0, a.vec4, v, flag);

  // chunk max and sum of exp
  float lm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4 * kExpVec; ++j) lm = fmaxf(lm, v[j]);
  const float Mc = block_max<kExpThreads>(lm, redz);
  float ls = 0.f;
  if (Mc > -INFINITY) {
#pragma unroll
    for (int j = 0; j < 4 * kExpVec; ++j) ls += (v[j] > -INFINITY) ? expf(v[j] - Mc) : 0.f;
  }
  const float Sc = block_sum<kExpThreads>(ls, redz);

  // per-warp top-k by repeated warp argmax (each lane pops its own best)
  unsigned consumed = 0;
  float bz = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < 4 * kExpVec; ++j) {
    const int id = chunk_id(c0, j, a.V);
    if (ranks_before(v[j], id, bz, bi)) { bz = v[j]; bi = id; }
  }
  for (int r = 0; r < k; ++r) {
    float z = bz;
    int id = bi;
    warp_best(z, id);
    if (lane == 0) { wz[warp][r] = z; wi[warp][r] = id; }
    if (id == bi && id != 0x7fffffff) {
#pragma unroll
      for (int j = 0; j < 4 * kExpVec; ++j)
        if (chunk_id(c0, j, a.V) == id) consumed |= 1u << j;
      bz = -INFINITY;
      bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 4 * kExpVec; ++j) {
        const int id2 = chunk_id(c0, j, a.V);
        if (!((consumed >> j) & 1u) && ranks_before(v[j], id2, bz, bi)) { bz = v[j]; bi = id2; }
      }
    }
  }
  __syncthreads();
  // block top-k: warp 0 merges the 8 warp lists
  float *prt = a.part + ((long long)row * a.nchunk + c) * (2 + 2 * k);
  if (warp == 0) {
    float cz[kExpThreads / 32];
    int ci[kExpThreads / 32];
#pragma unroll
    for (int q = 0; q < kExpThreads / 32; ++q) {
      const int idx = lane + 32 * q;
      if (idx < (kExpThreads / 32) * k) { cz[q] = wz[idx / k][idx % k]; ci[q] = wi[idx / k][idx % k]; }
      else { cz[q] = -INFINITY; ci[q] = 0x7fffffff; }
    }
    for (int r = 0; r < k; ++r) {
      float lz = -INFINITY;
      int li = 0x7fffffff, lq = -1;
#pragma unroll
      for (int q = 0; q < kExpThreads / 32; ++q)
        if (ranks_before(cz[q], ci[q], lz, li)) { lz = cz[q]; li = ci[q]; lq = q; }
      float z = lz;
      int id = li;
      warp_best(z, id);
      if (lane == 0) { prt[2 + 2 * r] = z; prt[3 + 2 * r] = __int_as_float(id); }
      if (id == li && lq >= 0 && id != 0x7fffffff) {
#pragma unroll
        for (int q = 0; q < kExpThreads / 32; ++q)
          if (q == lq) { cz[q] = -INFINITY; ci[q] = 0x7fffffff; }
      }
    }
    if (lane == 0) { prt[0] = Mc; prt[1] = Sc; }
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && c == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);

  // ---- last block of this row: merge the chunks, write the children ----
  if (!arrive_last(&a.row_cnt[row], (unsigned)a.nchunk, &sflag)) return;

  const float *rp = a.part + (long long)row * a.nchunk * (2 + 2 * k);
  float cm = -INFINITY, cs = 0.f;
  if (t < a.nchunk) { cm = ld_cg(rp + t * (2 + 2 * k)); cs = ld_cg(rp + t * (2 + 2 * k) + 1); }
  const float M = block_max<kExpThreads>(cm, redz);
  const float S = block_sum<kExpThreads>((t < a.nchunk && cm > -INFINITY) ? cs * expf(cm - M) : 0.f, redz);
  for (int i = t; i < a.nchunk * k; i += kExpThreads) {
    const int cc = i / k, r = i - cc * k;
    mz[i] = ld_cg(rp + cc * (2 + 2 * k) + 2 + 2 * r);
    mi[i] = __float_as_int(ld_cg(rp + cc * (2 + 2 * k) + 3 + 2 * r));
  }
  __syncthreads();
  float lz = -INFINITY;
  int li = 0x7fffffff;
  for (int i = t; i < a.nchunk * k; i += kExpThreads)
    if (ranks_before(mz[i], mi[i], lz, li)) { lz = mz[i]; li = mi[i]; }
  for (int r = 0; r < k; ++r) {
    float z = lz;
    int id = li;
    block_best<kExpThreads>(z, id, redz, redi);
    if (t == 0) { topz[r] = z; topi[r] = id; }
    if (id == li && id != 0x7fffffff) {  // the owner pops it and rescans its slots
      for (int i = t; i < a.nchunk * k; i += kExpThreads)
        if (mi[i] == id) { mz[i] = -INFINITY; mi[i] = 0x7fffffff; }
      lz = -INFINITY;
      li = 0x7fffffff;
      for (int i = t; i < a.nchunk * k; i += kExpThreads)
        if (ranks_before(mz[i], mi[i], lz, li)) { lz = mz[i]; li = mi[i]; }
    }
  }
  __syncthreads();
  if (t < k) {
    const float logS = (M > -INFINITY) ? logf(S) : 0.f;
    const float z = topz[t];
    const float lp = (M > -INFINITY && z > -INFINITY) ? (z - M) - logS : -INFINITY;
    const long long pkey = node < 0 ? 0ll : a.tree.cand_key[(long long)b * a.C + node];
    const int cid = a.base_next + s * k + t;
    const long long o = (long long)b * a.C + cid;
    const int tok = topi[t];
    a.tree.cand_tok[o] = (tok == 0x7fffffff) ? -1 : tok;
    a.tree.cand_parent[o] = node;
    a.tree.cand_lp[o] = lp;
    a.tree.cand_key[o] = add_keys(pkey, fixed_key(lp));
  }

  // ---- last row of this sequence: pick the next layer's frontier ----
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.m_l, &sflag)) return;
  if (a.m_next <= 0) return;
  const int width = a.m_l * k;  // <= 1024
  unsigned long long mine[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = t + q * kExpThreads;
    mine[q] = ~0ull;
    if (i < width) {
      const int id = a.base_next + i;
      mine[q] = rank_key(ld_cg(a.tree.cand_key + (long long)b * a.C + id), id);
    }
  }
  for (int r = 0; r < a.m_next; ++r) {
    unsigned long long lmin = ~0ull;
#pragma unroll
    for (int q = 0; q < 4; ++q) lmin = mine[q] < lmin ? mine[q] : lmin;
    const unsigned long long w = block_min_u64<kExpThreads>(lmin, red64);
    if (t == 0) sel[r] = (int)(w & ((1ull << kIdBits) - 1));
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (mine[q] == w) mine[q] = ~0ull;
  }
  __syncthreads();
  if (t < a.m) {
    int out = -1;
    if (t < a.m_next) {  // rank of sel[t] among the selected ids = its ascending slot
      int rank = 0;
      for (int j = 0; j < a.m_next; ++j) rank += sel[j] < sel[t];
      out = rank;
    }
    if (t < a.m_next) a.tree.frontier[b * a.m + out] = sel[t];
    else a.tree.frontier[b * a.m + t] = -1;
  }
}

// ---------------------------------------------------------------------------
// rerank + flatten
// ---------------------------------------------------------------------------
constexpr int kRrThreads = 1024;
constexpr int kRrBinBits = 11;
constexpr int kRrBins = 1 << kRrBinBits;    // two per thread at 1024 threads
constexpr int kRrBinCap = 64;               // keys of one bin ranked by counting

struct RerankArgs {
  int B, C, n, N, depth;
  int base[kMaxDepth + 2];
  et_tree tree;
  int32_t *dev_status;
  // optional (et_tree_rerank_mask): ancestor mask and position ids as well
  const int32_t *prefix_len;
  uint64_t *mask;
  int32_t *posids;
};

// Shared memory of one sequence's rerank (and of the fused mask).
struct RerankSmem {
  unsigned int hist[kRrBins];
  unsigned long long red_lo[32], red_hi[32], bin_keys[kRrBinCap];
  unsigned long long s_lo, s_hi, s_thr;
  int s_bin;
  unsigned int s_before, s_nb, s_cnt;
  short flat_of[kMaxC];
  unsigned char kept[kMaxC];
  int tmp[32];
  int row_par[kMaxN], row_dep[kMaxN];  // fused mask: parent row and depth of each flat row
};

// Ancestor bitmask of flat row i from its parent rows (parents precede
// children): bit j set iff row j is i or an ancestor of i.  Returns false on
// a parent that does not precede its child.
__device__ __forceinline__ bool ancestor_bits(const int *par, int i, uint64_t &w0, uint64_t &w1) {
  w0 = 0; w1 = 0;
  int j = i, steps = 0;
  while (j >= 0 && steps <= kMaxN) {  // parents have smaller rows: at most N steps
    if (j < 64) w0 |= 1ull << j; else w1 |= 1ull << (j - 64);
    const int p = par[j];
    if (p >= j) return false;
    j = p;
    ++steps;
  }
  return true;
}

// Exclusive prefix sum over the NT threads of a block (NT a multiple of 32,
// at most 1024); `total` gets the block's sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int *tmp, int &total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < NW ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s;  // inclusive prefix of warp totals
  }
  __syncthreads();
  total = tmp[NW - 1];
  const int before = w > 0 ? tmp[w - 1] : 0;
  __syncthreads();  // tmp may be reused by the next call
  return before + x - v;
}

// The n-th smallest of the C rank keys by histogram (keys are unique): a
// 2048-bin histogram over [min, max] puts it in one bin; that
// bin's keys are ranked by counting when few, else the bin's range is
// histogrammed again (each pass narrows the range by 2^11, so six passes
// reach single keys).  Marks the kept candidates in sm.kept.
template <int NT>
__device__ void rerank_select_hist(const RerankArgs &a, const unsigned long long (&rk)[kMaxC / NT], RerankSmem &sm) {
  constexpr int kPer = kMaxC / NT;
  constexpr int kHB = kRrBins / NT;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = a.C;
  unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (t + q * NT < C) {
      mn = rk[q] < mn ? rk[q] : mn;
      mx = rk[q] > mx ? rk[q] : mx;
    }
  }
  mn = warp_min_u64(mn);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = y > mx ? y : mx;
  }
  if (lane == 0) { sm.red_lo[warp] = mn; sm.red_hi[warp] = mx; }
  for (int i = t; i < kRrBins; i += NT) sm.hist[i] = 0u;
  if (t == 0) sm.s_cnt = 0u;
  __syncthreads();
  if (warp == 0) {
    mn = lane < NT / 32 ? sm.red_lo[lane] : ~0ull;
    mx = lane < NT / 32 ? sm.red_hi[lane] : 0ull;
    mn = warp_min_u64(mn);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, mx, o);
      mx = y > mx ? y : mx;
    }
    if (lane == 0) { sm.s_lo = mn; sm.s_hi = mx; sm.s_thr = ~0ull; }
  }
  __syncthreads();
  unsigned long long lo = sm.s_lo, hi = sm.s_hi;
  unsigned int remaining = (unsigned)a.n;  // 1-based rank of the wanted key among keys in [lo, hi]
  for (int pass = 0; pass < 7; ++pass) {
    const unsigned long long range = hi - lo;
    const int bits = range ? 64 - __clzll((long long)range) : 0;
    const int shift = bits > kRrBinBits ? bits - kRrBinBits : 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      if (t + q * NT < C && rk[q] >= lo && rk[q] <= hi) atomicAdd(&sm.hist[(rk[q] - lo) >> shift], 1u);
    __syncthreads();
    unsigned int h[kHB], hs = 0;  // this thread's kHB consecutive bins
#pragma unroll
    for (int e = 0; e < kHB; ++e) { h[e] = sm.hist[kHB * t + e]; hs += h[e]; }
    int total;
    const unsigned int excl = (unsigned)block_excl_scan<NT>((int)hs, sm.tmp, total);
    if (excl < remaining && remaining <= excl + hs) {
      unsigned int before = excl;
#pragma unroll
      for (int e = 0; e < kHB; ++e) {
        if (before < remaining && remaining <= before + h[e]) {
          sm.s_bin = kHB * t + e;
          sm.s_before = before;
          sm.s_nb = h[e];
        }
        before += h[e];
      }
    }
    __syncthreads();
    const int B = sm.s_bin;
    const unsigned int nb = sm.s_nb;
    remaining -= sm.s_before;
    const unsigned long long blo = lo + ((unsigned long long)B << shift);
    const unsigned long long bhi = shift ? (hi - blo < (1ull << shift) - 1 ? hi : blo + ((1ull << shift) - 1)) : blo;
    if (nb <= (unsigned)kRrBinCap) {  // always so for shift == 0 (one key per value)
#pragma unroll
      for (int q = 0; q < kPer; ++q)
        if (t + q * NT < C && rk[q] >= blo && rk[q] <= bhi) sm.bin_keys[atomicAdd(&sm.s_cnt, 1u)] = rk[q];
      __syncthreads();
      if (t < (int)nb) {
        const unsigned long long mine = sm.bin_keys[t];
        unsigned int r = 0;
        for (unsigned int j = 0; j < nb; ++j) r += sm.bin_keys[j] < mine ? 1u : 0u;
        if (r + 1 == remaining) sm.s_thr = mine;
      }
      __syncthreads();
      break;
    }
    lo = blo;
    hi = bhi;
    for (int i = t; i < kRrBins; i += NT) sm.hist[i] = 0u;
    __syncthreads();
  }
  const unsigned long long thr = sm.s_thr;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int id = t + q * NT;
    if (id < C) sm.kept[id] = rk[q] <= thr ? 1 : 0;
  }
  __syncthreads();
}

// Flatten the kept candidates (ids ascending -> rows 1..n) and write the
// flat arrays; with a.mask set, the ancestor mask and positions as well.
template <int NT>
__device__ void flatten_and_mask(const RerankArgs &a, int b, const int (&pre_tok)[kMaxC / NT],
                                 const int (&pre_par)[kMaxC / NT], RerankSmem &sm) {
  constexpr int kPer = kMaxC / NT;
  const int t = threadIdx.x;
  const int C = a.C;
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int id = kPer * t + j;
    cnt += (id < C && sm.kept[id]) ? 1 : 0;
  }
  int total;
  int run = block_excl_scan<NT>(cnt, sm.tmp, total);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int id = kPer * t + j;
    if (id < C) sm.flat_of[id] = sm.kept[id] ? (short)(1 + run++) : (short)-1;
  }
  __syncthreads();
  const long long fo = (long long)b * a.N;
  int bad = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int id = kPer * t + j;
    if (id >= C || !sm.kept[id]) continue;
    const int row = sm.flat_of[id];
    if (row < 1 || row >= a.N) { bad = 1; continue; }  // never write outside the flat arrays
    const int p = pre_par[j];
    int prow = 0;
    if (p >= 0) {
      prow = (p < C) ? sm.flat_of[p] : -1;
      if (prow < 0) { bad = 1; prow = 0; }
    }
    int depth = 1;
    for (int l = 1; l <= a.depth; ++l)
      if (id >= a.base[l]) depth = l;
    a.tree.flat_node[fo + row] = id;
    a.tree.flat_tok[fo + row] = pre_tok[j];
    a.tree.flat_parent[fo + row] = prow;
    a.tree.flat_depth[fo + row] = depth;
    sm.row_par[row] = prow;
    sm.row_dep[row] = depth;
  }
  if (bad) flag_status(a.dev_status, ET_DEV_DISCONNECTED);
  if (t == 0) {
    a.tree.flat_node[fo] = -1;
    a.tree.flat_tok[fo] = a.tree.root_tok ? a.tree.root_tok[b] : -1;
    a.tree.flat_parent[fo] = -1;
    a.tree.flat_depth[fo] = 0;
    sm.row_par[0] = -1;
    sm.row_dep[0] = 0;
  }
  if (!a.mask) return;
  // ---- fused: ancestor mask + position ids of the rows just written ----
  __syncthreads();
  const int N = a.N, W = (N + 63) >> 6;
  if (t < N) {
    uint64_t w0, w1;
    const bool ok = ancestor_bits(sm.row_par, t, w0, w1);
    uint64_t *mrow = a.mask + ((long long)b * N + t) * W;
    mrow[0] = w0;
    if (W > 1) mrow[1] = w1;
    a.posids[(long long)b * N + t] = a.prefix_len[b] + sm.row_dep[t];
    if (!ok) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  }
}

// Rerank + flatten of sequence b by one block of NT threads (reranking
// phase of the EAGLE-2 article): keep the n candidates with the smallest
// rank keys ((key desc, id asc): equal values keep the shallower node, so the
// kept tree is connected), rows 1..n = kept ids ascending; with a.mask set,
// the ancestor mask and position ids of the rows just written as well.
template <int NT>
__device__ void rerank_sequence(const RerankArgs &a, int b, RerankSmem &sm) {
  constexpr int kPer = kMaxC / NT;     // candidates per thread
  const int t = threadIdx.x;
  const int C = a.C;

  unsigned long long rk[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int id = t + q * NT;
    rk[q] = id < C ? rank_key(ld_cg(a.tree.cand_key + (long long)b * C + id), id) : ~0ull;
  }
  if (t < kMaxN) { sm.row_par[t] = 0; sm.row_dep[t] = 0; }  // rows a broken tree leaves unwritten
  // the token and parent of this thread's flatten ids, fetched now (they are
  // needed only after the selection)
  int pre_tok[kPer], pre_par[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int id = kPer * t + j;
    pre_tok[j] = id < C ? ld_cg(a.tree.cand_tok + (long long)b * C + id) : -1;  // L2: the candidates may have
    pre_par[j] = id < C ? ld_cg(a.tree.cand_parent + (long long)b * C + id) : -1;  // been written in this launch
  }
  rerank_select_hist<NT>(a, rk, sm);
  // flatten: kept ids ascending -> rows 1..n
  flatten_and_mask<NT>(a, b, pre_tok, pre_par, sm);
}

__global__ void __launch_bounds__(kRrThreads) k_rerank(RerankArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  __shared__ RerankSmem sm;
  rerank_sequence<kRrThreads>(a, blockIdx.x, sm);
}

// ---------------------------------------------------------------------------
// ancestor mask + position ids
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxN) k_mask_posids(int N, const int32_t *flat_parent, const int32_t *flat_depth,
                                                      const int32_t *prefix_len, uint64_t *mask, int32_t *posids,
                                                      int32_t *dev_status) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  __shared__ int par[kMaxN];
  const int b = blockIdx.x, i = threadIdx.x;
  const int W = (N + 63) >> 6;
  if (i < N) par[i] = flat_parent[(long long)b * N + i];
  __syncthreads();
  if (i >= N) return;
  uint64_t w0, w1;
  const int bad = ancestor_bits(par, i, w0, w1) ? 0 : 1;
  uint64_t *mrow = mask + ((long long)b * N + i) * W;
  mrow[0] = w0;
  if (W > 1) mrow[1] = w1;
  posids[(long long)b * N + i] = prefix_len[b] + flat_depth[(long long)b * N + i];
  if (bad) flag_status(dev_status, ET_DEV_BAD_INDEX);
}

struct ExpandRowArgs {
  const float *logits;
  long long row_stride;
  const int32_t *row_of_node;
  int vec4;
  int B, V, k, m, C, layer, m_l, base_next, m_next;
  et_tree tree;
  int32_t *dev_status;
  unsigned int *seq_cnt;  // [B]
};

// ---------------------------------------------------------------------------
// expand, one thread-block cluster per expanded row (V <= 32768): CTA q of the
// cluster owns logits [4096 q, 4096 q + 4096) (16 per thread).  Each warp
// finds the exact top-k of its 512 logits and their (max, sum of exp) and
// stores both straight into the leader's (rank 0) shared memory; after one
// cluster barrier the leader's first warp merges the 8R sorted warp lists
// into the row's top-k, normalises, and writes the children.  The last row
// of a sequence then picks the next frontier among the first m children of
// every row.  Spreading a row over up to 8 SMs gives the load 8x the memory
// parallelism of one block per row; keeping every step after the load inside
// one warp (no block-wide select) keeps the chain short.
// ---------------------------------------------------------------------------
constexpr int kClThreads = 256;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClVec = 4;
constexpr int kClSpan = kClThreads * 4 * kClVec;   // 4096 logits per CTA
constexpr int kClMaxCtas = 8;
constexpr int kClMaxV = kClSpan * kClMaxCtas;      // 32768
constexpr int kClLists = kClMaxCtas * kClWarps;    // warp lists of one row

// ---- warp-level selection ----
__device__ __forceinline__ unsigned int f32_ord(float x) {  // ascending with x (no NaN)
  const unsigned int u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_f32(unsigned int o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ float warp_max_f(float x) { return ord_f32(__reduce_max_sync(0xffffffffu, f32_ord(x))); }
__device__ __forceinline__ float warp_min_f(float x) { return ord_f32(__reduce_min_sync(0xffffffffu, f32_ord(x))); }
// How many lanes of the warp hold a larger value than this lane's x (four
// independent counters: a short dependency chain).
__device__ __forceinline__ int lanes_above(float x) {
  int c4[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 32; ++j) c4[j & 3] += __shfl_sync(0xffffffffu, x, j) > x ? 1 : 0;
  return (c4[0] + c4[1]) + (c4[2] + c4[3]);
}
// exclusive prefix sum over the warp of c, 0 <= c < 2^BITS
template <int BITS>
__device__ __forceinline__ int warp_excl_prefix(int c) {
  unsigned int lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  int pos = 0;
#pragma unroll
  for (int bit = 0; bit < BITS; ++bit) pos += __popc(__ballot_sync(0xffffffffu, (c >> bit) & 1) & lt) << bit;
  return pos;
}
// how many of cand[0 .. nc) are below mine (broadcast reads, eight independent per round)
__device__ __forceinline__ int count_below(const unsigned long long *cand, int nc, unsigned long long mine) {
  int r = 0, j = 0;
  for (; j + 8 <= nc; j += 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u) r += cand[j + u] < mine ? 1 : 0;
  }
  for (; j < nc; ++j) r += cand[j] < mine ? 1 : 0;
  return r;
}
// cand[0 .. nc) (nc <= 32, distinct) -> lane r < n returns the r-th smallest, other lanes ~0
__device__ __forceinline__ unsigned long long warp_rank_small(unsigned long long *cand, int nc, int n) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const unsigned long long mine = lane < nc ? cand[lane] : ~0ull;
  const int r = count_below(cand, nc, mine);
  __syncwarp();
  if (lane < nc && r < n) cand[r] = mine;
  __syncwarp();
  const unsigned long long out = lane < n ? cand[lane] : ~0ull;
  __syncwarp();
  return out;
}

// The warp's (max, sum of exp(z - max)) over its lanes' NV logits each,
// with the lane's own maximum in lane_max (EAGLE-2 article, expansion phase:
// the softmax normaliser of a node's draft distribution).  NaN counts as -inf
// and +inf as FLT_MAX (flag set); padding must already be -inf.  The common
// case costs a max and an exponential a value: fmaxf skips NaN, and a NaN or
// +inf leaves a NaN in the lane's sum (inf - inf), so only a warp whose sum
// turned NaN, or whose maximum is -inf (nothing to show a NaN), sanitises
// its values and starts again.
template <int NV>
__device__ __forceinline__ float2 warp_row_stats(float (&v)[NV], float &lane_max, int &flag) {
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < NV; ++e) m = fmaxf(m, v[e]);
  float Mw = warp_max_f(m);
  float sum = 0.f;
  if (Mw > -INFINITY) {
#pragma unroll
    for (int e = 0; e < NV; ++e) sum += exp_fast(v[e] - Mw);
  }
  if (__any_sync(0xffffffffu, sum != sum || Mw == -INFINITY)) {
    m = -INFINITY;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      v[e] = sanitize_logit(v[e], flag);
      m = fmaxf(m, v[e]);
    }
    Mw = warp_max_f(m);
    sum = 0.f;
    if (Mw > -INFINITY) {
#pragma unroll
      for (int e = 0; e < NV; ++e) sum += exp_fast(v[e] - Mw);
    }
  }
  lane_max = m;
  return make_float2(Mw, warp_sum(sum));
}

// The warp's best values at or above tau, at most k of them (value desc,
// id asc), as ascending (value, id) keys: lane r < n returns the r-th, the
// other lanes ~0.  v: sanitised values (no NaN), id_of(e): the id of the
// lane's e-th value (distinct over the warp); k <= 32; cand: 32 keys of warp
// scratch; n: how many are returned.  Usually none or a few values reach tau: they are ranked by
// counting; more than 32 (ties, or a warp holding many of the row's best
// values) take k rounds of a warp argmin, whose k keys all reach tau then.
template <int NV, typename IdOf>
__device__ __forceinline__ unsigned long long warp_best_at_least(const float (&v)[NV], float lane_max, IdOf id_of,
                                                                 float tau, int k, unsigned long long *cand, int &n) {
  static_assert(NV <= 32, "a lane's values fit one 32-bit mask");
  constexpr int kCountBits = NV < 32 ? 5 : 6;  // a lane's count, 0 .. NV
  const int lane = threadIdx.x & 31;
  if (!__any_sync(0xffffffffu, lane_max >= tau)) {  // most warps of a row
    n = 0;
    return ~0ull;
  }
  unsigned int msk = 0u;
#pragma unroll
  for (int e = 0; e < NV; ++e) msk |= (v[e] >= tau ? 1u : 0u) << e;
  const int c = __popc(msk);
  const int nc = (int)__reduce_add_sync(0xffffffffu, (unsigned int)c);
  if (nc == 0) {
    n = 0;
    return ~0ull;
  }
  if (nc <= 32) {
    int pos = warp_excl_prefix<kCountBits>(c);
    if (c) {
#pragma unroll
      for (int e = 0; e < NV; ++e)
        if ((msk >> e) & 1u) cand[pos++] = zid_key(v[e], id_of(e));
    }
    n = nc < k ? nc : k;
    return warp_rank_small(cand, nc, n);
  }
  unsigned long long out = ~0ull, lb = ~0ull;
  unsigned int used = 0u;
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const unsigned long long x = zid_key(v[e], id_of(e));
    lb = x < lb ? x : lb;
  }
  for (int r = 0; r < k; ++r) {
    const unsigned long long m = warp_min_u64(lb);
    if (lane == r) out = m;
    if (lb == m) {
      lb = ~0ull;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const unsigned long long x = zid_key(v[e], id_of(e));
        if (x == m) used |= 1u << e;
        if (!((used >> e) & 1u) && x < lb) lb = x;
      }
    }
  }
  __syncwarp();
  n = k;
  return out;
}

// Shared memory of one expanding CTA.  Every CTA holds every warp's (max,
// sum) pair of the row (by layer parity: a pair of the next layer may land
// while the leader still reads this one); the leader also holds each warp's
// candidates and their count.
struct ExpandClSmem {
  float2 pairs[2][kClLists];                      // (max, sum of exp) of warp w of CTA q at 8 q + w
  unsigned long long lists[kClLists * kMaxTopk];  // leader: warp (q, w)'s candidates, ascending, at (8 q + w) * k
  int counts[kClLists];                           // leader: how many
  unsigned long long cand[kClWarps][32];          // per-warp selection scratch
  float2 norm;                                     // leader: the row's (max, log of the sum of exp)
};

__device__ __forceinline__ void cl_st_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// One row's logits in the CTA's registers: 16 per thread, float4 loads
// when the row is 16-byte aligned; ids >= V (and a missing row) are -inf.
__device__ __forceinline__ void load_row_span(const float *zrow, int base, int V, int vec4, float (&v)[4 * kClVec]) {
  const int t = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kClVec; ++u) {
    const int e0 = base + u * kClThreads * 4 + t * 4;
    if (zrow && vec4 && e0 + 3 < V) {
      const float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < V) ? __ldcs(zrow + e0 + j) : -INFINITY;
    }
  }
}

// Every warp of every CTA of the row's cluster (EAGLE-2 article, expansion
// phase: the top-k children of a node by draft confidence).  1: sanitise its
// 512 logits; their max and sum of exp go to every CTA of the cluster (the
// caller has completed the previous cluster phase: every block has started,
// or every block is done with the previous layer).  2: after one cluster barrier
// every warp takes, from the R x 8 warp maxima, the k-th largest lane
// maximum (each lane holds two warps' maxima), tau: k distinct values of the
// row reach it, so only values >= tau can be among the row's top k.  3: each
// warp sends its best values >= tau (at most k, ascending) to the leader.
// The caller then arrives on the barrier that releases these stores.
__device__ __forceinline__ void row_warp_part(float (&v)[4 * kClVec], int base, int V, int k, int par, ExpandClSmem &sh,
                                              int &flag) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int q = (int)cl_rank(), R = (int)gridDim.x;
  float lane_max;
  const float2 st = warp_row_stats(v, lane_max, flag);  // ids >= V are padding (-inf)
  const int list = q * kClWarps + warp;
  if (lane < R) cl_st_f32x2(cl_map(&sh.pairs[par][list], (uint32_t)lane), st.x, st.y);
  cl_arrive();
  cl_wait();  // every warp's pair is in every block
  const int nl = R * kClWarps;
  const float lm = fmaxf(lane < nl ? sh.pairs[par][lane].x : -INFINITY, lane + 32 < nl ? sh.pairs[par][lane + 32].x : -INFINITY);
  const int above = lanes_above(lm);
  const float tau = warp_min_f(above < k ? lm : INFINITY);
  int n = 0;
  const unsigned long long key = warp_best_at_least<4 * kClVec>(
      v, lane_max, [&](int e) { return (unsigned int)(base + (e >> 2) * kClThreads * 4 + t * 4 + (e & 3)); }, tau,
      k, sh.cand[warp], n);
  if (lane < n) cl_st_u64(cl_map(&sh.lists[list * k + lane], 0), key);
  if (lane == 0) cl_st_s32(cl_map(&sh.counts[list], 0), n);
}

// The leader's first two warps, once every warp's candidates have landed:
// warp 1 forms the row's normaliser (log-softmax, from the warp pairs) while
// warp 0 selects the row's top-k children, then writes them with their path
// keys (EAGLE-2 article: expansion phase; the value of a path is the product
// of confidences, here a sum of fixed-point log-probs).  The candidates
// number at least k (every warp among the k holding the largest maxima sends
// its maximum); a few more usually: ranked by counting.  More than 32: k
// rounds of the smallest list head.  nl: warp lists of the row (8 R).
__device__ __forceinline__ void row_leader_part(const float2 *pairs, const unsigned long long *lists,
                                                const int *counts, unsigned long long *cand, float2 *norm, int nl,
                                                int k, int V, const et_tree &tree, long long o0, int parent,
                                                long long pkey) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) == 1) {
    const float2 pa = lane < nl ? pairs[lane] : make_float2(-INFINITY, 0.f);
    const float2 pb = lane + 32 < nl ? pairs[lane + 32] : make_float2(-INFINITY, 0.f);
    const float M = warp_max_f(fmaxf(pa.x, pb.x));
    float part = 0.f;
    if (M > -INFINITY) {
      part = (pa.x > -INFINITY ? pa.y * expf(pa.x - M) : 0.f) + (pb.x > -INFINITY ? pb.y * expf(pb.x - M) : 0.f);
    }
    const float S = warp_sum(part);
    if (lane == 0) *norm = make_float2(M, (M > -INFINITY) ? logf(S) : 0.f);
    asm volatile("bar.sync 1, 64;" ::: "memory");  // with warp 0: the normaliser is in
    return;
  }
  const int la = lane, lb = lane + 32;
  const int ca = la < nl ? counts[la] : 0, cb = lb < nl ? counts[lb] : 0;
  const int nc = (int)__reduce_add_sync(0xffffffffu, (unsigned int)(ca + cb));
  unsigned long long key_r;
  if (nc <= 32) {
    int pos = warp_excl_prefix<7>(ca + cb);
    for (int j = 0; j < ca; ++j) cand[pos++] = lists[la * k + j];
    for (int j = 0; j < cb; ++j) cand[pos++] = lists[lb * k + j];
    key_r = warp_rank_small(cand, nc, k);
  } else {
    int pa_ = 0, pb_ = 0;
    unsigned long long ha = ca > 0 ? lists[la * k] : ~0ull, hb = cb > 0 ? lists[lb * k] : ~0ull;
    key_r = ~0ull;
    for (int r = 0; r < k; ++r) {
      const unsigned long long m = warp_min_u64(ha < hb ? ha : hb);
      if (lane == r) key_r = m;
      if (ha == m) {
        ++pa_;
        ha = pa_ < ca ? lists[la * k + pa_] : ~0ull;
      } else if (hb == m) {
        ++pb_;
        hb = pb_ < cb ? lists[lb * k + pb_] : ~0ull;
      }
    }
  }
  asm volatile("bar.sync 1, 64;" ::: "memory");  // with warp 1
  const float M = norm->x, logS = norm->y;
  if (lane < k) {
    const float z = zid_value(key_r);
    const int id = (int)zid_id(key_r);
    const float lp = (M > -INFINITY && z > -INFINITY) ? (z - M) - logS : -INFINITY;
    const long long o = o0 + lane;
    tree.cand_tok[o] = id < V ? id : -1;
    tree.cand_parent[o] = parent;
    tree.cand_lp[o] = lp;
    tree.cand_key[o] = add_keys(pkey, fixed_key(lp));
  }
}

// The last row of sequence b to finish a layer picks the next layer's
// frontier: the m_next best children of the layer by rank key (EAGLE-2
// article, expansion phase: the top-m nodes by path value expand next),
// written in ascending id order, the unused slots -1.  A child at position e
// of its row has e better siblings, so only the first m_next of every row can
// rank below m_next, and among them ranks below m_next are exact.  Every
// thread of the block takes part.
template <int NT>
__device__ __forceinline__ void pick_next_frontier(const et_tree &tree, int b, int C, int k, int m, int m_l,
                                                   int m_next, int base_next, unsigned long long *fl, int *sel,
                                                   const int32_t *rmap = nullptr, int *rowof = nullptr,
                                                   int *frow = nullptr) {
  const int t = threadIdx.x;
  const int nk = k < m_next ? k : m_next;
  const int P = m_l * nk;  // <= 1024
  for (int c = t; c < P; c += NT) {
    const int rs = c / nk, e = c - rs * nk;
    const int id = base_next + rs * k + e;
    fl[c] = rank_key(ld_cg(tree.cand_key + (long long)b * C + id), id);
    if (rmap) rowof[c] = rmap[(long long)b * (C + 1) + id + 1];  // the table row, in the same round
  }
  __syncthreads();
  block_select<NT>(fl, P, m_next, [&](int r, unsigned long long key_r) {
    sel[r] = (int)(key_r & ((1ull << kIdBits) - 1));
  });
  __syncthreads();
  if (t < m) {
    if (t < m_next) {
      int slot = 0;
      const int mine = sel[t];
      for (int j = 0; j < m_next; ++j) slot += sel[j] < mine ? 1 : 0;
      tree.frontier[b * m + slot] = mine;
      if (rmap) {
        const int rs = (mine - base_next) / k, e = (mine - base_next) - rs * k;
        frow[b * kMaxM + slot] = rowof[rs * nk + e];
      }
    } else {
      tree.frontier[b * m + t] = -1;
    }
  }
}

__global__ void __launch_bounds__(kClThreads) k_expand_cl(ExpandRowArgs a) {
  __shared__ ExpandClSmem sh;
  __shared__ unsigned long long fl[kMaxM * kMaxTopk];  // the last leader: frontier candidates
  __shared__ int sel[kMaxM];
  __shared__ int last;
  const int t = threadIdx.x, warp = t >> 5;
  const int R = gridDim.x;                 // CTAs per row = cluster size
  const int q = (int)cl_rank();
  const int row = blockIdx.y;
  const int b = row / a.m_l, s = row - b * a.m_l;
  const int k = a.k;
  cl_arrive_relaxed();  // this block has started (waited on before any remote store)
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead

  int flag = 0, bad = 0;
  int node = -1;
  if (a.layer > 0) {
    node = a.tree.frontier[b * a.m + s];
    if (node < 0 || node >= a.C) bad = 1;
  }
  const float *zrow = nullptr;
  if (!bad) {
    long long r = a.row_of_node ? (long long)a.row_of_node[(long long)b * (a.C + 1) + node + 1] : (long long)row;
    if (r < 0) bad = 1;
    else zrow = a.logits + r * a.row_stride;
  }
  const int base = q * kClSpan;
  float v[4 * kClVec];
  load_row_span(zrow, base, a.V, a.vec4, v);
  // the parent's path key, fetched while the logits are in flight
  const long long pkey = (q == 0 && warp == 0 && node >= 0 && !bad) ? ld_cg(a.tree.cand_key + (long long)b * a.C + node)
                                                                    : 0ll;
  cl_wait();  // every block of the cluster runs
  row_warp_part(v, base, a.V, k, 0, sh, flag);
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  cl_arrive();  // release the candidates
  if (q != 0) return;
  cl_wait();

  // ---- the leader's first two warps: the row's top-k and normaliser; write the children ----
  if (warp < 2)
    row_leader_part(sh.pairs[0], sh.lists, sh.counts, sh.cand[0], &sh.norm, R * kClWarps, k, a.V, a.tree,
                    (long long)b * a.C + a.base_next + s * k, node, pkey);
  if (a.m_next <= 0) return;  // last layer: no frontier to pick

  // ---- the last row of this sequence picks the next frontier ----
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.m_l, &last)) return;
  pick_next_frontier<kClThreads>(a.tree, b, a.C, a.k, a.m, a.m_l, a.m_next, a.base_next, fl, sel);
}

// ---------------------------------------------------------------------------
// expand, one 1024-thread block per expanded row (V <= 32768), for layers of
// many rows.  The cluster kernel needs 8 blocks of 64 registers a thread per
// row, so only 4 of its blocks fit an SM and a layer of a few hundred rows
// runs in several waves of that kernel's latency chain (load, cluster
// barrier, threshold, cluster barrier, leader).  Here one block holds the
// whole row in registers (32 logits a thread, the same 128-bit loads) and
// every exchange is a block barrier: each of the 32 warps forms its (max,
// sum of exp) and, after one barrier, the k-th largest warp maximum, tau;
// it sends its best values >= tau (at most k) to shared lists; after a
// second barrier warps 0 and 1 select and normalise exactly as the cluster
// leader does.  The children and the frontier are those of k_expand_cl; the
// log-probs may differ in the last bits (the sum of exp is taken in another
// order).
// ---------------------------------------------------------------------------
constexpr int kWdThreads = 1024;
constexpr int kWdWarps = kWdThreads / 32;
constexpr int kWdVec = 8;  // float4 loads a thread: 32 logits
static_assert(kWdThreads * 4 * kWdVec == kClMaxV, "one block spans the widest row of the cluster kernel");

struct ExpandWdSmem {
  float2 pairs[kWdWarps];                          // (max, sum of exp) of warp w
  unsigned long long lists[kWdWarps * kMaxTopk];  // warp w's candidates, ascending, at w * k
  int counts[kWdWarps];                            // how many
  unsigned long long cand[kWdWarps][32];           // per-warp selection scratch
  unsigned long long fl[kMaxM * kMaxTopk];         // the sequence's last row: frontier candidates
  int rowof[kMaxM * kMaxTopk];                     // their table rows (the work-queue build)
  int sel[kMaxM];
  float2 norm;                                     // the row's (max, log of the sum of exp)
  int last;
};

// One row of the expansion by a whole 1024-thread block (every thread calls
// it): the row's logits into registers, the warp statistics, the threshold,
// each warp's candidates, then warps 0 and 1 write the k children at o0..
// (parent `parent`, path keys from *pkey_src, 0 when null).  zrow null: a
// missing row, all -inf.  Ends with the children written by warp 0 (no
// barrier after them).
__device__ __forceinline__ void wide_row(const float *zrow, int V, int vec4, int k, const et_tree &tree, long long o0,
                                         int parent, const int64_t *pkey_src, int32_t *dev_status,
                                         ExpandWdSmem &sh) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // thread t holds logits 4096 u + 4 t + j, u < 8, j < 4; ids >= V (and a missing row) are -inf
  float v[4 * kWdVec];
#pragma unroll
  for (int u = 0; u < kWdVec; ++u) {
    const int e0 = u * kWdThreads * 4 + t * 4;
    if (zrow && vec4 && e0 + 3 < V) {
      const float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < V) ? __ldcs(zrow + e0 + j) : -INFINITY;
    }
  }
  // the parent's path key, fetched while the logits are in flight
  const long long pkey = (warp == 0 && pkey_src) ? ld_cg(pkey_src) : 0ll;
  int flag = 0;
  float lane_max;
  const float2 st = warp_row_stats(v, lane_max, flag);
  if (lane == 0) sh.pairs[warp] = st;
  __syncthreads();
  // tau: the k-th largest warp maximum (lane j holds warp j's); k distinct
  // values of the row reach it, so only values >= tau can be in the top k
  const float lm = sh.pairs[lane].x;
  const int above = lanes_above(lm);
  const float tau = warp_min_f(above < k ? lm : INFINITY);
  int n = 0;
  const unsigned long long key = warp_best_at_least<4 * kWdVec>(
      v, lane_max, [&](int e) { return (unsigned int)((e >> 2) * kWdThreads * 4 + t * 4 + (e & 3)); }, tau, k,
      sh.cand[warp], n);
  if (lane < n) sh.lists[warp * k + lane] = key;
  if (lane == 0) sh.counts[warp] = n;
  if (flag) flag_status(dev_status, ET_DEV_NONFINITE);
  __syncthreads();
  if (warp < 2) row_leader_part(sh.pairs, sh.lists, sh.counts, sh.cand[0], &sh.norm, kWdWarps, k, V, tree, o0, parent, pkey);
}

__global__ void __launch_bounds__(kWdThreads) k_expand_wd(ExpandRowArgs a) {
  __shared__ ExpandWdSmem sh;
  const int t = threadIdx.x;
  const int row = blockIdx.x;
  const int b = row / a.m_l, s = row - b * a.m_l;
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead

  int bad = 0;
  int node = -1;
  if (a.layer > 0) {
    node = a.tree.frontier[b * a.m + s];
    if (node < 0 || node >= a.C) bad = 1;
  }
  const float *zrow = nullptr;
  if (!bad) {
    long long r = a.row_of_node ? (long long)a.row_of_node[(long long)b * (a.C + 1) + node + 1] : (long long)row;
    if (r < 0) bad = 1;
    else zrow = a.logits + r * a.row_stride;
  }
  wide_row(zrow, a.V, a.vec4, a.k, a.tree, (long long)b * a.C + a.base_next + s * a.k, node,
           (node >= 0 && !bad) ? a.tree.cand_key + (long long)b * a.C + node : nullptr, a.dev_status, sh);
  if (bad && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  if (a.m_next <= 0) return;  // last layer: no frontier to pick
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.m_l, &sh.last)) return;
  pick_next_frontier<kWdThreads>(a.tree, b, a.C, a.k, a.m, a.m_l, a.m_next, a.base_next, sh.fl, sh.sel);
}

// ---------------------------------------------------------------------------
// The whole draft tree in one launch: the expansion phase layer after layer,
// then the reranking phase with the attention mask and positions (EAGLE-2
// article).  One cluster of ceil(V / 4096) CTAs per (sequence, frontier
// slot) stays resident for all D layers: slot s of sequence b expands the
// s-th frontier node of every layer that expands more than s nodes (layer 0:
// the root, in slot 0), with the same per-row work as k_expand_cl.  Each row
// of a layer arrives on the layer's counter once its children are written.
// A cluster of the next layer waits (bounded spin) until every row of the
// previous layer has arrived, then picks the frontier itself -- the top m of
// the first min(k, m) children of each previous row, as k_expand_cl's last
// leader does -- fetching the candidates' keys and table rows in one round,
// and takes its slot's node (slot 0 also writes the frontier array).  The
// sequence's last row of the final layer re-arms the layer counters; the
// rerank, mask and positions follow as one more launch (k_rerank, whose 1024
// threads select faster than one 256-thread block could here).  Every
// cluster must be resident
// at once (they wait on one another): the host launches this kernel only
// when the occupancy calculator says they all fit.  Data written inside the
// launch (candidates) is read through L2 (ld.cg), not L1, which other SMs'
// writes do not update.
// ---------------------------------------------------------------------------
struct BuildArgs {
  const float *logits;
  long long row_stride;
  const int32_t *row_of_node;
  int vec4;
  int B, V, k, m, C, D, slots;  // slots: clusters per sequence (the widest layer's expanded rows)
  int expanded[kMaxDepth];
  int base[kMaxDepth + 2];
  et_tree tree;
  int32_t *dev_status;
  unsigned int *layer_cnt;  // [B][kMaxDepth] rows of each layer whose children are written; back to 0 at the end
  long long wait_cycles;    // bound of a wait for the previous layer (et_set_wait_limit)
  int rerank_here;          // one more cluster per sequence reranks the tree inside this launch
  int n, N;                 // kept nodes, flat rows
  const int32_t *prefix_len;
  uint64_t *mask;           // nullable: no mask and positions
  int32_t *posids;
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct BuildPick {
  unsigned long long fl[kMaxM * kMaxTopk];  // frontier candidates (rank keys)
  int rowof[kMaxM * kMaxTopk];              // their table rows
  int sel[kMaxM];
  long long s_row;
  int s_node;
};

// The rerank inside k_tree_build, by the leader block of one more cluster per
// sequence: as each layer completes, its children are merged into the
// running top-n (top-n of a union = top-n of the running top-n and the new
// candidates; rank keys are unique, so the result is exact), each key ranked
// by counting; after the last layer the kept ids, sorted by id, become flat
// rows 1..n (reranking phase of the EAGLE-2 article), with the mask and the
// positions.  The merges run beside the layers, off their critical path.
struct RerankRoleSmem {
  unsigned long long ks[256];        // running top-n, then the layer's candidates
  unsigned long long keep[kMaxN];    // the new running top-n, by rank
  int keep_tok[kMaxN], keep_par[kMaxN];  // their tokens and parents (carried, so the flatten loads nothing)
  int ids[kMaxN];                    // kept candidate ids
  short flat_of[kMaxC];              // flat row of each kept id, -1 otherwise
  int row_par[kMaxN], row_dep[kMaxN];
};

__device__ void rerank_role(const BuildArgs &a, int b, unsigned int *cnt, RerankRoleSmem &sm) {
  const int t = threadIdx.x;
  const int C = a.C, n = a.n, N = a.N;
  int nk = 0;  // keys in the running top-n
  for (int layer = 0; layer < a.D; ++layer) {
    const int m_l = a.expanded[layer], width = m_l * a.k, base_next = a.base[layer + 1];
    if (t == 0 && ld_acquire_u32(cnt + layer) < (unsigned)m_l) {
      const long long t0 = clock64();
      while (ld_acquire_u32(cnt + layer) < (unsigned)m_l) {
        if (clock64() - t0 > a.wait_cycles) {
          flag_status(a.dev_status, ET_DEV_TIMEOUT);
          break;
        }
      }
    }
    __syncthreads();
    const int P = nk + width;  // <= 256 (checked by the host)
    unsigned long long mine = ~0ull;
    int mtok = -1, mpar = -1;
    if (t < nk) {
      mine = sm.keep[t];
      mtok = sm.keep_tok[t];
      mpar = sm.keep_par[t];
    } else if (t < P) {  // the key, token and parent in one round
      const int id = base_next + (t - nk);
      const long long o = (long long)b * C + id;
      mine = rank_key(ld_cg(a.tree.cand_key + o), id);
      mtok = ld_cg(a.tree.cand_tok + o);
      mpar = ld_cg(a.tree.cand_parent + o);
    }
    __syncthreads();  // every running key read before ks is rewritten
    sm.ks[t] = mine;
    __syncthreads();
    if (t < P) {
      int c4[4] = {0, 0, 0, 0};  // independent counters: short dependency chains
      int j = 0;
      for (; j + 4 <= P; j += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) c4[u] += sm.ks[j + u] < mine ? 1 : 0;
      }
      for (; j < P; ++j) c4[0] += sm.ks[j] < mine ? 1 : 0;
      const int below = (c4[0] + c4[1]) + (c4[2] + c4[3]);
      if (below < n) {  // ranks are unique: the running list stays sorted
        sm.keep[below] = mine;
        sm.keep_tok[below] = mtok;
        sm.keep_par[below] = mpar;
      }
    }
    nk = P < n ? P : n;
    __syncthreads();
  }
  // kept ids -> flat rows 1..n in ascending id order
  for (int i = t; i < C; i += kClThreads) sm.flat_of[i] = -1;
  if (t < kMaxN) { sm.row_par[t] = 0; sm.row_dep[t] = 0; }
  if (t < nk) sm.ids[t] = (int)(sm.keep[t] & ((1ull << kIdBits) - 1));
  __syncthreads();
  int myrow = -1, myid = -1;
  if (t < nk) {
    myid = sm.ids[t];
    int c4[4] = {0, 0, 0, 0};
    int j = 0;
    for (; j + 4 <= nk; j += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) c4[u] += sm.ids[j + u] < myid ? 1 : 0;
    }
    for (; j < nk; ++j) c4[0] += sm.ids[j] < myid ? 1 : 0;
    myrow = 1 + (c4[0] + c4[1]) + (c4[2] + c4[3]);
    sm.flat_of[myid] = (short)myrow;
  }
  __syncthreads();
  const long long fo = (long long)b * N;
  int bad = 0;
  if (t < nk && myrow < N) {
    const int tok = sm.keep_tok[t];  // the merges carried them with the key
    const int p = sm.keep_par[t];
    int prow = 0;
    if (p >= 0) {
      prow = p < C ? sm.flat_of[p] : -1;
      if (prow < 0) { bad = 1; prow = 0; }
    }
    int depth = 1;
    for (int l = 1; l <= a.D; ++l)
      if (myid >= a.base[l]) depth = l;
    a.tree.flat_node[fo + myrow] = myid;
    a.tree.flat_tok[fo + myrow] = tok;
    a.tree.flat_parent[fo + myrow] = prow;
    a.tree.flat_depth[fo + myrow] = depth;
    sm.row_par[myrow] = prow;
    sm.row_dep[myrow] = depth;
  }
  if (bad) flag_status(a.dev_status, ET_DEV_DISCONNECTED);
  if (t == 0) {
    a.tree.flat_node[fo] = -1;
    a.tree.flat_tok[fo] = a.tree.root_tok ? a.tree.root_tok[b] : -1;
    a.tree.flat_parent[fo] = -1;
    a.tree.flat_depth[fo] = 0;
    sm.row_par[0] = -1;
    sm.row_dep[0] = 0;
    for (int l = 0; l < a.D; ++l) cnt[l] = 0u;  // every wait of this sequence is over: re-arm for the next call
  }
  if (!a.mask) return;
  __syncthreads();
  const int W = (N + 63) >> 6;
  if (t < N) {
    uint64_t w0, w1;
    const bool ok = ancestor_bits(sm.row_par, t, w0, w1);
    uint64_t *mrow = a.mask + ((long long)b * N + t) * W;
    mrow[0] = w0;
    if (W > 1) mrow[1] = w1;
    a.posids[(long long)b * N + t] = a.prefix_len[b] + sm.row_dep[t];
    if (!ok) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  }
}

union BuildSmem {
  ExpandClSmem e;
  RerankRoleSmem r;
};

__global__ void __launch_bounds__(kClThreads) k_tree_build(BuildArgs a) {
  __shared__ BuildSmem sh;
  __shared__ BuildPick pk;
  ExpandClSmem &sh_e = sh.e;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int R = gridDim.x;  // CTAs per row = cluster size
  const int q = (int)cl_rank();
  const int per_seq = a.slots + (a.rerank_here ? 1 : 0);
  const int b = blockIdx.y / per_seq, s = blockIdx.y - b * per_seq;
  const int k = a.k;
  unsigned int *cnt = a.layer_cnt + (long long)b * kMaxDepth;
  cl_arrive_relaxed();  // phase 0: this block has started (waited on before any remote store)
  pdl_wait();           // returns at once: this kernel is launched stream-ordered (see et_tree_build)
  pdl_trigger();        // every block of this grid is resident before a dependent can launch
  if (s == a.slots) {   // the rerank cluster: its leader alone works
    if (q == 0) rerank_role(a, b, cnt, sh.r);
    return;
  }
  cl_wait();  // every block of the cluster runs (before any remote store)

  for (int layer = 0; layer < a.D; ++layer) {
    const int m_l = a.expanded[layer];
    if (s >= m_l) continue;  // this slot has no node to expand in this layer (the whole cluster skips it)
    const int base_next = a.base[layer + 1];
    int node = -1, bad = 0;
    long long row = (long long)b * m_l + s;  // the table row without a row map
    if (layer > 0) {
      // every row of the previous layer has written its children
      const int m_prev = a.expanded[layer - 1];
      if (t == 0 && ld_acquire_u32(cnt + layer - 1) < (unsigned)m_prev) {
        const long long t0 = clock64();
        while (ld_acquire_u32(cnt + layer - 1) < (unsigned)m_prev) {
          if (clock64() - t0 > a.wait_cycles) {  // never expected: report, go on (outputs invalid)
            flag_status(a.dev_status, ET_DEV_TIMEOUT);
            break;
          }
        }
      }
      __syncthreads();
      const int base_l = a.base[layer];
      const int nk = k < m_l ? k : m_l;
      const int P = m_prev * nk;
      for (int c = t; c < P; c += kClThreads) {
        const int rs = c / nk, e = c - rs * nk;
        const int id = base_l + rs * k + e;
        pk.fl[c] = rank_key(ld_cg(a.tree.cand_key + (long long)b * a.C + id), id);
        if (a.row_of_node) pk.rowof[c] = a.row_of_node[(long long)b * (a.C + 1) + id + 1];
      }
      __syncthreads();
      block_select<kClThreads>(pk.fl, P, m_l, [&](int r, unsigned long long key_r) {
        pk.sel[r] = (int)(key_r & ((1ull << kIdBits) - 1));
      });
      __syncthreads();
      if (t < m_l) {  // slots hold the picked ids in ascending order
        const int mine = pk.sel[t];
        int slot = 0;
        for (int j = 0; j < m_l; ++j) slot += pk.sel[j] < mine ? 1 : 0;
        if (slot == s) {
          pk.s_node = mine;
          const int rs = (mine - base_l) / k, e = (mine - base_l) - rs * k;
          pk.s_row = a.row_of_node ? pk.rowof[rs * nk + e] : row;
        }
        if (s == 0 && q == 0) a.tree.frontier[b * a.m + slot] = mine;
      } else if (s == 0 && q == 0 && t < a.m) {
        a.tree.frontier[b * a.m + t] = -1;
      }
      __syncthreads();
      node = pk.s_node;
      row = pk.s_row;
      if (node < 0 || node >= a.C) bad = 1;
    } else if (a.row_of_node) {
      row = a.row_of_node[(long long)b * (a.C + 1)];  // the root
    }
    const float *zrow = nullptr;
    if (!bad && row >= 0) zrow = a.logits + row * a.row_stride;
    else bad = 1;
    const int base = q * kClSpan;
    int flag = 0;
    float v[4 * kClVec];
    load_row_span(zrow, base, a.V, a.vec4, v);
    const long long pkey = (q == 0 && warp == 0 && node >= 0 && !bad) ? ld_cg(a.tree.cand_key + (long long)b * a.C + node)
                                                                      : 0ll;
    row_warp_part(v, base, a.V, k, layer & 1, sh_e, flag);
    if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
    if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    cl_arrive();  // release the candidates
    cl_wait();    // every block's candidates have landed in the leader (and every block is done with this layer)
    if (q == 0 && warp < 2)
      row_leader_part(sh_e.pairs[layer & 1], sh_e.lists, sh_e.counts, sh_e.cand[0], &sh_e.norm, R * kClWarps, k, a.V,
                      a.tree, (long long)b * a.C + base_next + s * k, node, pkey);
    if (q == 0 && warp == 0) {
      __threadfence();
      __syncwarp();  // every child of this row is written
      if (lane == 0) {
        const bool last = atomicAdd(cnt + layer, 1u) == (unsigned)(m_l - 1);  // the next layer may count this row
        // the sequence's last row of the final layer (when no rerank cluster
        // follows the layers): every wait of this sequence is over, re-arm
        // the counters for the next call
        if (last && layer + 1 == a.D && !a.rerank_here)
          for (int l = 0; l < a.D; ++l) cnt[l] = 0u;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The whole draft tree in one launch for batches whose clusters do not all
// fit k_tree_build (EAGLE-2 article: expansion layer after layer, then the
// reranking phase with the attention mask and positions).  Persistent
// 1024-thread blocks take work items from a counter: one item per expanded
// row, in layer-major order (layer, then sequence, then frontier slot), each
// expanded as k_expand_wd expands a row.  An item of layer l > 0 waits
// (bounded spin) only for its own sequence's layer-l frontier, so the layers
// of different sequences overlap and no layer waits for a whole-grid
// boundary.  The last row of a sequence's layer (arrival counter) picks the
// next frontier and publishes it with a release flag; the last row of its
// final layer reranks the sequence in the same block (the rerank kernel's
// code, 1024 threads) and clears the sequence's flags.  No deadlock
// whatever the residency: an item waits only on items of earlier layers,
// which blocks that are already running took before it.  The last block to
// run out of items re-arms the item counter.
// ---------------------------------------------------------------------------
struct FlowArgs {
  const float *logits;
  long long row_stride;
  const int32_t *row_of_node;
  int vec4;
  int V, k, m, C, D;
  int expanded[kMaxDepth];
  int base[kMaxDepth + 2];
  int item0[kMaxDepth + 1];  // first item of each layer; item0[D] = the number of items
  et_tree tree;
  int32_t *dev_status;
  unsigned int *layer_cnt;   // [B][kMaxDepth] rows of a layer whose children are written (the last re-arms it)
  unsigned int *ready;       // [B][kMaxDepth] 1 once the layer's frontier is written (cleared by the rerank)
  unsigned int *work;        // [2] next item, blocks out of items (both back to 0 at the end)
  int *frow;                 // [B][kMaxM] table row of each frontier slot (with row_of_node)
  long long wait_cycles;     // bound of a wait for a frontier (et_set_wait_limit)
  RerankArgs rr;             // the rerank, mask and positions of each sequence
};

union FlowSmem {
  ExpandWdSmem e;
  RerankSmem r;
};

__device__ __forceinline__ void st_release_u32(unsigned int *p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kWdThreads) k_tree_flow(FlowArgs a) {
  __shared__ FlowSmem sh;
  __shared__ int s_item, s_last;  // outside the union: read after the barriers that end a phase
  const int t = threadIdx.x;
  pdl_wait();     // returns at once: this kernel is launched stream-ordered (see et_tree_build)
  pdl_trigger();  // every block of this grid is resident before a dependent can launch
  const int total = a.item0[a.D];
  for (;;) {
    if (t == 0) s_item = (int)atomicAdd(a.work, 1u);
    __syncthreads();
    const int i = s_item;
    if (i >= total) break;
    int l = 0;
    while (l + 1 < a.D && i >= a.item0[l + 1]) ++l;
    const int m_l = a.expanded[l];
    const int j = i - a.item0[l], b = j / m_l, s = j - b * m_l;
    unsigned int *cnt = a.layer_cnt + (long long)b * kMaxDepth;
    unsigned int *rdy = a.ready + (long long)b * kMaxDepth;
    int node = -1, bad = 0;
    if (l > 0) {
      // this sequence's frontier of layer l is written
      if (t == 0 && ld_acquire_u32(rdy + l) == 0u) {
        const long long t0 = clock64();
        while (ld_acquire_u32(rdy + l) == 0u) {
          if (clock64() - t0 > a.wait_cycles) {  // never expected: report, go on (outputs invalid)
            flag_status(a.dev_status, ET_DEV_TIMEOUT);
            break;
          }
        }
      }
      __syncthreads();
    }
    // the node and its table row (written in this launch by the picker: read through L2, in one round)
    long long r = (long long)b * m_l + s;
    if (l > 0) {
      node = ld_cg(a.tree.frontier + b * a.m + s);
      if (a.row_of_node) r = ld_cg(a.frow + b * kMaxM + s);
      if (node < 0 || node >= a.C) bad = 1;
    } else if (a.row_of_node) {
      r = a.row_of_node[(long long)b * (a.C + 1)];  // the root
    }
    const float *zrow = nullptr;
    if (!bad) {
      if (r < 0) bad = 1;
      else zrow = a.logits + r * a.row_stride;
    }
    wide_row(zrow, a.V, a.vec4, a.k, a.tree, (long long)b * a.C + a.base[l + 1] + s * a.k, node,
             (node >= 0 && !bad) ? a.tree.cand_key + (long long)b * a.C + node : nullptr, a.dev_status, sh.e);
    if (bad && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    if (arrive_last(cnt + l, (unsigned)m_l, &s_last)) {
      if (l + 1 < a.D) {
        pick_next_frontier<kWdThreads>(a.tree, b, a.C, a.k, a.m, m_l, a.expanded[l + 1], a.base[l + 1], sh.e.fl,
                                       sh.e.sel, a.row_of_node, sh.e.rowof, a.frow);
        __syncthreads();  // every frontier slot is written
        if (t == 0) {
          __threadfence();
          st_release_u32(rdy + l + 1, 1u);
        }
      } else {
        // every item of this sequence is done: rerank it, then clear its flags
        rerank_sequence<kWdThreads>(a.rr, b, sh.r);
        if (t < a.D) rdy[t] = 0u;
      }
    }
    __syncthreads();  // s_item and the shared memory are free for the next item
  }
  if (t == 0) {
    __threadfence();
    if (atomicAdd(a.work + 1, 1u) == gridDim.x - 1) {  // every block is out of items
      a.work[0] = 0u;
      a.work[1] = 0u;
    }
  }
}

}  // namespace et

using namespace et;

// ---------------------------------------------------------------------------
// workspace layout shared by et_tree_expand and et_verify_accept
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct TreeWs {
  size_t cnt_bytes, part_off, rowstat_off, dq_off, total;
  int rows;  // max rows of one launch
};

static int nchunk_of(int V) { return (V + kExpChunk - 1) / kExpChunk; }

static TreeWs tree_ws_layout(const et_tree_cfg *cfg) {
  TreeWs w{};
  const int N = cfg->n + 1;
  const int nch = nchunk_of(cfg->V);
  const int rows = cfg->B * (cfg->m > N ? cfg->m : N);
  w.rows = rows;
  // counters: [rows] per row, [B] per sequence, [B][kMaxDepth] per layer and [B][kMaxDepth]
  // frontier flags (et_tree_build), 2 item counters and [B][kMaxM] frontier table rows
  // (et_tree_build's work-queue form)
  w.cnt_bytes = align256(sizeof(unsigned int) *
                         (size_t)(rows + cfg->B + 2 * (size_t)cfg->B * kMaxDepth + 2 + (size_t)cfg->B * kMaxM));
  const size_t exp_part = sizeof(float) * (size_t)cfg->B * cfg->m * nch * (2 + 2 * cfg->topk);
  const size_t ver_part = sizeof(float) * (size_t)cfg->B * N * nch * 2;
  w.part_off = w.cnt_bytes;
  const size_t part = align256(exp_part > ver_part ? exp_part : ver_part);
  w.rowstat_off = w.part_off + part;
  // draft-q acceptance: per flat row q's max and sum and the residual pairs (c, F)
  w.dq_off = w.rowstat_off + align256(sizeof(float) * 2 * (size_t)cfg->B * N);
  w.total = w.dq_off + align256(sizeof(float) * 8 * (size_t)cfg->B * N);
  return w;
}

extern "C" size_t et_tree_workspace_size(const et_tree_cfg *cfg) {
  Geometry g;
  if (!make_geometry(cfg, &g)) return 0;
  return tree_ws_layout(cfg).total;
}

// used by et_verify.cu; not part of the ABI
// A logit table may sit in device memory or in page-locked host memory that
// the device addresses (the kernels then read only the rows they need over
// the host link: NVLink-C2C on Grace-Blackwell).  Writes the address the
// kernels use into *dev; returns 0, launching nothing, for memory the device
// cannot address (pageable host memory) or a pointer the runtime does not know;
// 1 for device (or managed) memory, 2 for page-locked host memory.
extern "C" __attribute__((visibility("hidden"))) int et_internal_table_ptr(const void *p, const void **dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *dev = p;
    return 1;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer) {
    *dev = at.devicePointer;
    return 2;
  }
  return 0;
}

static bool table_ptr(const float *p, const float **dev) {
  const void *d = nullptr;
  if (!et_internal_table_ptr(p, &d)) return false;
  *dev = static_cast<const float *>(d);
  return true;
}

extern "C" __attribute__((visibility("hidden"))) size_t et_internal_tree_ws(const et_tree_cfg *cfg, size_t *cnt_bytes, size_t *part_off,
                                      size_t *rowstat_off, size_t *dq_off) {
  TreeWs w = tree_ws_layout(cfg);
  *dq_off = w.dq_off;
  *cnt_bytes = w.cnt_bytes;
  *part_off = w.part_off;
  *rowstat_off = w.rowstat_off;
  return w.total;
}

extern "C" int32_t et_num_candidates(const et_tree_cfg *cfg) {
  Geometry g;
  return make_geometry(cfg, &g) ? g.C : -1;
}

extern "C" int32_t et_layer_expanded(const et_tree_cfg *cfg, int32_t layer) {
  Geometry g;
  if (!make_geometry(cfg, &g) || layer < 0 || layer >= cfg->depth) return -1;
  return g.expanded[layer];
}

extern "C" int32_t et_layer_base(const et_tree_cfg *cfg, int32_t layer) {
  Geometry g;
  if (!make_geometry(cfg, &g) || layer < 1 || layer > cfg->depth) return -1;
  return g.base[layer];
}

// one block per expanded row; same arguments as the chunked kernel
// Which kernel expands a layer when V <= 32768 (et_set_expand_kernel): the
// cluster kernel spreads a row over ceil(V / 4096) SMs, which shortens each
// row's load when the layer has few rows; one block per row saves the
// cluster barriers and runs more rows at once when it has many.
static std::atomic<int> g_expand_kernel{ET_EXPAND_AUTO};
constexpr int kWdMinRows = 64;  // auto: one block per row from this many rows of a layer

static et_status launch_expand_row(const ExpandArgs &c, cudaStream_t stream) {
  ExpandRowArgs a;
  a.logits = c.logits; a.row_stride = c.row_stride; a.row_of_node = c.row_of_node; a.vec4 = c.vec4;
  a.B = c.B; a.V = c.V; a.k = c.k; a.m = c.m; a.C = c.C; a.layer = c.layer; a.m_l = c.m_l;
  a.base_next = c.base_next; a.m_next = c.m_next;
  a.tree = c.tree; a.dev_status = c.dev_status; a.seq_cnt = c.seq_cnt;
  const int rows = c.B * c.m_l;
  const int which = g_expand_kernel.load(std::memory_order_relaxed);
  if (which == ET_EXPAND_BLOCK || (which == ET_EXPAND_AUTO && rows >= kWdMinRows))
    return et_launch(k_expand_wd, dim3(rows, 1, 1), dim3(kWdThreads, 1, 1), 0, stream, 0, a);
  // one cluster of ceil(V / 4096) CTAs per expanded row
  const int R = (c.V + kClSpan - 1) / kClSpan;
  return et_launch(k_expand_cl, dim3(R, rows, 1), dim3(kClThreads, 1, 1), 0, stream, R, a);
}

extern "C" int32_t et_set_expand_kernel(int32_t which) {
  if (which != ET_EXPAND_AUTO && which != ET_EXPAND_CLUSTER && which != ET_EXPAND_BLOCK) return -1;
  return g_expand_kernel.exchange(which);
}

static bool tree_ptrs_ok(const et_tree *t) {
  return t && t->cand_tok && t->cand_parent && t->cand_lp && t->cand_key && t->frontier;
}

extern "C" et_status et_tree_expand(const et_tree_cfg *cfg, int32_t layer, const float *logits, int64_t row_stride,
                                    const int32_t *row_of_node, et_tree *tree, int32_t *dev_status, void *ws,
                                    size_t ws_bytes, et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(layer < 0 || layer >= cfg->depth, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!logits || row_stride < cfg->V || !tree_ptrs_ok(tree), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  const TreeWs w = tree_ws_layout(cfg);
  ET_RETURN_IF(!ws || ws_bytes < w.total || !et_aligned(ws, 256), ET_ERR_WORKSPACE);
  const int m_l = g.expanded[layer];
  ET_RETURN_IF((long long)cfg->B * m_l > 65535, ET_ERR_UNSUPPORTED);
  ET_RETURN_IF(!table_ptr(logits, &logits), ET_ERR_INVALID_ARG);  // device, or page-locked host memory
  ExpandArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.row_of_node = row_of_node;
  a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
  a.B = cfg->B; a.V = cfg->V; a.k = cfg->topk; a.m = cfg->m; a.C = g.C; a.layer = layer; a.m_l = m_l;
  a.base_next = g.base[layer + 1];
  a.m_next = (layer + 1 < cfg->depth) ? g.expanded[layer + 1] : 0;
  a.nchunk = nchunk_of(cfg->V);
  a.tree = *tree;
  a.dev_status = dev_status;
  unsigned char *base = static_cast<unsigned char *>(ws);
  a.row_cnt = reinterpret_cast<unsigned int *>(base);
  a.seq_cnt = a.row_cnt + w.rows;
  a.part = reinterpret_cast<float *>(base + w.part_off);
  if (cfg->V <= kClMaxV) return launch_expand_row(a, (cudaStream_t)stream);
  dim3 grid(a.nchunk, cfg->B * m_l);
  const size_t smem = (size_t)a.nchunk * a.k * (sizeof(float) + sizeof(int));
  return et_launch(k_expand, grid, dim3(kExpThreads), smem, (cudaStream_t)stream, 0, a);
}

static RerankArgs rerank_args(const et_tree_cfg *cfg, const Geometry &g, const et_tree *tree, int32_t *dev_status,
                              const int32_t *prefix_len, uint64_t *mask, int32_t *posids) {
  RerankArgs a;
  a.B = cfg->B; a.C = g.C; a.n = cfg->n; a.N = cfg->n + 1; a.depth = cfg->depth;
  for (int l = 0; l < kMaxDepth + 2; ++l) a.base[l] = (l <= cfg->depth + 1) ? g.base[l] : 0x7fffffff;
  a.base[0] = 0;
  a.tree = *tree;
  a.dev_status = dev_status;
  a.prefix_len = prefix_len;
  a.mask = mask;
  a.posids = posids;
  return a;
}

static et_status launch_rerank(const et_tree_cfg *cfg, et_tree *tree, int32_t *dev_status, const int32_t *prefix_len,
                               uint64_t *mask, int32_t *posids, et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!tree || !tree->cand_tok || !tree->cand_parent || !tree->cand_key || !tree->flat_node ||
                   !tree->flat_tok || !tree->flat_parent || !tree->flat_depth,
               ET_ERR_INVALID_ARG);
  const RerankArgs a = rerank_args(cfg, g, tree, dev_status, prefix_len, mask, posids);
  return et_launch(k_rerank, dim3(cfg->B), dim3(kRrThreads), 0, (cudaStream_t)stream, 0, a);
}

extern "C" et_status et_tree_rerank(const et_tree_cfg *cfg, et_tree *tree, int32_t *dev_status, et_stream_t stream) {
  return launch_rerank(cfg, tree, dev_status, nullptr, nullptr, nullptr, stream);
}

extern "C" et_status et_tree_rerank_mask(const et_tree_cfg *cfg, et_tree *tree, const int32_t *prefix_len,
                                         uint64_t *mask, int32_t *posids, int32_t *dev_status, et_stream_t stream) {
  ET_RETURN_IF(!prefix_len || !mask || !posids, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(mask, 8), ET_ERR_INVALID_ARG);
  return launch_rerank(cfg, tree, dev_status, prefix_len, mask, posids, stream);
}

// The whole tree in one cluster launch (k_tree_build) when every one of its
// clusters fits on the GPU at once; otherwise in one work-queue launch
// (k_tree_flow), or, past one cluster (V > 32768), as D expansion launches
// and the fused rerank launch.
static int tree_build_fits(int clusters, int R) {
  static std::mutex mu;
  static int cached_dev = -1, cached_R = -1, cached_n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev != cached_dev || R != cached_R) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(R, clusters, 1);
    lc.blockDim = dim3(kClThreads, 1, 1);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)R;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    lc.attrs = &attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)k_tree_build, &lc) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached_dev = dev;
    cached_R = R;
    cached_n = n;
  }
  return clusters <= cached_n;
}

// Blocks of k_tree_flow that the current device holds at once (cached per device).
static long long flow_blocks() {
  static std::mutex mu;
  static int cached_dev = -1;
  static long long cached_n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev != cached_dev) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_tree_flow, kWdThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    cached_dev = dev;
    cached_n = (long long)sms * (per_sm > 0 ? per_sm : 1);
  }
  return cached_n;
}

extern "C" et_status et_tree_build(const et_tree_cfg *cfg, const float *logits, int64_t row_stride,
                                   const int32_t *row_of_node, et_tree *tree, const int32_t *prefix_len,
                                   uint64_t *mask, int32_t *posids, int32_t *dev_status, void *ws, size_t ws_bytes,
                                   et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!logits || row_stride < cfg->V || !tree_ptrs_ok(tree) || !et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!tree->flat_node || !tree->flat_tok || !tree->flat_parent || !tree->flat_depth, ET_ERR_INVALID_ARG);
  ET_RETURN_IF((mask || posids) && (!mask || !posids || !prefix_len || !et_aligned(mask, 8)), ET_ERR_INVALID_ARG);
  const TreeWs w = tree_ws_layout(cfg);
  ET_RETURN_IF(!ws || ws_bytes < w.total || !et_aligned(ws, 256), ET_ERR_WORKSPACE);
  const float *const logits_in = logits;  // the per-layer form resolves the table itself
  ET_RETURN_IF(!table_ptr(logits, &logits), ET_ERR_INVALID_ARG);  // device, or page-locked host memory
  int slots = 1, widest = 0;
  for (int l = 0; l < cfg->depth; ++l) {
    slots = g.expanded[l] > slots ? g.expanded[l] : slots;
    widest = g.expanded[l] * cfg->topk > widest ? g.expanded[l] * cfg->topk : widest;
  }
  const int R = (cfg->V + kClSpan - 1) / kClSpan;
  const bool rerank_here = cfg->n + widest <= kClThreads;  // every merge ranks at most one key per thread
  const long long clusters = (long long)cfg->B * (slots + (rerank_here ? 1 : 0));
  const int which = g_expand_kernel.load(std::memory_order_relaxed);
  if (cfg->V <= kClMaxV && which != ET_EXPAND_BLOCK && clusters <= 65535 && tree_build_fits((int)clusters, R)) {
    BuildArgs a;
    a.logits = logits;
    a.row_stride = row_stride;
    a.row_of_node = row_of_node;
    a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
    a.B = cfg->B; a.V = cfg->V; a.k = cfg->topk; a.m = cfg->m; a.C = g.C; a.D = cfg->depth; a.slots = slots;
    for (int l = 0; l < kMaxDepth; ++l) a.expanded[l] = l < cfg->depth ? g.expanded[l] : 0;
    for (int l = 0; l < kMaxDepth + 2; ++l) a.base[l] = (l <= cfg->depth + 1) ? g.base[l] : 0x7fffffff;
    a.tree = *tree;
    a.dev_status = dev_status;
    unsigned char *base = static_cast<unsigned char *>(ws);
    a.layer_cnt = reinterpret_cast<unsigned int *>(base) + w.rows + cfg->B;  // the per-layer counters
    a.wait_cycles = et_wait_limit_cycles();
    a.rerank_here = rerank_here ? 1 : 0;
    a.n = cfg->n;
    a.N = cfg->n + 1;
    a.prefix_len = prefix_len;
    a.mask = mask;
    a.posids = posids;
    // A plain stream-ordered launch: as a programmatic dependent, the grid's
    // clusters were placed while the previous kernel still held the SMs, and
    // the build ran about 15 us slower behind attention or acceptance on
    // GB300 (no slowdown behind another tree build or a non-programmatic
    // kernel).  The kernel still triggers its own dependents early.
    const et_status st = et_launch_ex(false, k_tree_build, dim3(R, (unsigned)clusters, 1), dim3(kClThreads, 1, 1),
                                      0, (cudaStream_t)stream, R, a);
    if (st != ET_OK || rerank_here) return st;
    return launch_rerank(cfg, tree, dev_status, prefix_len, mask, posids, stream);
  }
  if (cfg->V <= kClMaxV && which != ET_EXPAND_CLUSTER) {  // the clusters do not all fit: the work-queue form
    static_assert(kWdThreads == kRrThreads, "the flow blocks run the rerank's code");
    FlowArgs a;
    a.logits = logits;
    a.row_stride = row_stride;
    a.row_of_node = row_of_node;
    a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
    a.V = cfg->V; a.k = cfg->topk; a.m = cfg->m; a.C = g.C; a.D = cfg->depth;
    long long items = 0;
    for (int l = 0; l <= kMaxDepth; ++l) {
      a.item0[l] = (int)items;
      if (l < cfg->depth) items += (long long)cfg->B * g.expanded[l];
    }
    ET_RETURN_IF(items > 0x7fffffffll - 4 * 1024 * 1024, ET_ERR_UNSUPPORTED);
    for (int l = 0; l < kMaxDepth; ++l) a.expanded[l] = l < cfg->depth ? g.expanded[l] : 0;
    for (int l = 0; l < kMaxDepth + 2; ++l) a.base[l] = (l <= cfg->depth + 1) ? g.base[l] : 0x7fffffff;
    a.tree = *tree;
    a.dev_status = dev_status;
    unsigned int *counters = reinterpret_cast<unsigned int *>(ws);
    a.layer_cnt = counters + w.rows + cfg->B;
    a.ready = a.layer_cnt + (size_t)cfg->B * kMaxDepth;
    a.work = a.ready + (size_t)cfg->B * kMaxDepth;
    a.frow = reinterpret_cast<int *>(a.work + 2);
    a.wait_cycles = et_wait_limit_cycles();
    a.rr = rerank_args(cfg, g, tree, dev_status, prefix_len, mask, posids);
    // one block per SM can hold (64 registers x 1024 threads); more would only queue
    const int grid = (int)(items < flow_blocks() ? items : flow_blocks());
    // stream-ordered, as k_tree_build (blocks spin on flags that other blocks set)
    return et_launch_ex(false, k_tree_flow, dim3(grid, 1, 1), dim3(kWdThreads, 1, 1), 0, (cudaStream_t)stream, 0, a);
  }
  for (int l = 0; l < cfg->depth; ++l) {
    const et_status st = et_tree_expand(cfg, l, logits_in, row_stride, row_of_node, tree, dev_status, ws, ws_bytes,
                                        stream);
    if (st != ET_OK) return st;
  }
  return launch_rerank(cfg, tree, dev_status, prefix_len, mask, posids, stream);
}

extern "C" int32_t et_tree_build_launches(const et_tree_cfg *cfg) {
  Geometry g;
  if (!make_geometry(cfg, &g)) return -1;
  int slots = 1, widest = 0;
  for (int l = 0; l < cfg->depth; ++l) {
    slots = g.expanded[l] > slots ? g.expanded[l] : slots;
    widest = g.expanded[l] * cfg->topk > widest ? g.expanded[l] * cfg->topk : widest;
  }
  const int R = (cfg->V + kClSpan - 1) / kClSpan;
  const bool rerank_here = cfg->n + widest <= kClThreads;
  const long long clusters = (long long)cfg->B * (slots + (rerank_here ? 1 : 0));
  const int which = g_expand_kernel.load(std::memory_order_relaxed);
  if (cfg->V <= kClMaxV && which != ET_EXPAND_BLOCK && clusters <= 65535 && tree_build_fits((int)clusters, R))
    return rerank_here ? 1 : 2;
  if (cfg->V <= kClMaxV && which != ET_EXPAND_CLUSTER) return 1;  // the work-queue form
  return cfg->depth + 1;
}

extern "C" et_status et_tree_mask_posids(const et_tree_cfg *cfg, const et_tree *tree, const int32_t *prefix_len,
                                         uint64_t *mask, int32_t *posids, et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!tree || !tree->flat_parent || !tree->flat_depth || !prefix_len || !mask || !posids,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(mask, 8), ET_ERR_INVALID_ARG);
  return et_launch(k_mask_posids, dim3(cfg->B), dim3(kMaxN), 0, (cudaStream_t)stream, 0, cfg->n + 1,
                   (const int32_t *)tree->flat_parent, (const int32_t *)tree->flat_depth, prefix_len, mask, posids,
                   (int32_t *)nullptr);
}

extern "C" et_status et_workspace_init(void *ws, size_t ws_bytes, et_stream_t stream) {
  if (!ws_bytes) return ET_OK;
  ET_RETURN_IF(!ws, ET_ERR_WORKSPACE);
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? ET_OK : ET_ERR_CUDA;
}

extern "C" const char *et_status_string(et_status s) {
  switch (s) {
    case ET_OK: return "ok";
    case ET_ERR_INVALID_ARG: return "invalid argument";
    case ET_ERR_UNSUPPORTED: return "unsupported shape";
    case ET_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ET_ERR_CUDA: return "CUDA launch or runtime error";
    case ET_ERR_TIMEOUT: return "bounded device wait gave up";
  }
  return "unknown status";
}

extern "C" int32_t et_abi_version(void) { return ET_ABI_VERSION; }

// ---------------------------------------------------------------------------
// the bound of device waits (a diagnostic: small values make waits expire)
// ---------------------------------------------------------------------------
static constexpr long long kDefaultWaitCycles = 1ll << 32;  // ~2 s at 2 GHz
static std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

long long et_wait_limit_cycles() { return g_wait_cycles.load(std::memory_order_relaxed); }

extern "C" int64_t et_set_wait_limit(int64_t cycles) {
  return g_wait_cycles.exchange(cycles > 0 ? (long long)cycles : kDefaultWaitCycles);
}

// ---------------------------------------------------------------------------
// et_tree_expand_noalloc: et_tree_expand with its scratch in a static device
// array, for callers that must not allocate device memory themselves.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace et {
// Scratch of et_tree_expand_noalloc: per-chunk partial results and arrival
// counters.  Every GPU that loads this library holds one copy until exit.
constexpr size_t kExpandScratchBytes = 4u << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_expand_scratch[kExpandScratchBytes];

// The array's name is only a host-side stand-in in host code.  Its device
// address belongs to the module loaded in one CUDA context, so it is looked up
// (cudaGetSymbolAddress, with that context's device current) the first time a
// context calls, and kept per context.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
static CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    cudaGetLastError();
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

constexpr int kMaxScratchCtx = 64;
static std::mutex g_scratch_mu;
static CUcontext g_scratch_ctx[kMaxScratchCtx];
static void *g_scratch_ptr[kMaxScratchCtx];
static int g_scratch_n = 0, g_scratch_next = 0;

static et_status expand_scratch(void **out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const CtxGetCurrentFn cur = ctx_get_current();
  CUcontext ctx = nullptr;
  if (cur && cur(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  for (int i = 0; ctx && i < g_scratch_n; ++i)
    if (g_scratch_ctx[i] == ctx) {
      *out = g_scratch_ptr[i];
      return ET_OK;
    }
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_expand_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return ET_ERR_CUDA;
  }
  if (cur && !ctx && cur(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // the look-up made the primary context current
  if (ctx) {  // remember it (the oldest entry makes room when the table is full)
    const int slot = g_scratch_n < kMaxScratchCtx ? g_scratch_n++ : (g_scratch_next++ % kMaxScratchCtx);
    g_scratch_ctx[slot] = ctx;
    g_scratch_ptr[slot] = p;
  }
  *out = p;
  return ET_OK;
}
}  // namespace et

extern "C" et_status et_tree_expand_noalloc(const et_tree_cfg *cfg, int32_t layer, const float *logits,
                                            int64_t row_stride, const int32_t *row_of_node, et_tree *tree,
                                            int32_t *dev_status, et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(layer < 0 || layer >= cfg->depth, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!logits || row_stride < cfg->V || !tree_ptrs_ok(tree), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  const int m_l = g.expanded[layer];
  ET_RETURN_IF((long long)cfg->B * m_l > 65535, ET_ERR_UNSUPPORTED);
  // this launch's scratch: counters (rows + sequences), then the per-chunk partials
  const int rows = cfg->B * m_l;
  const int nchunk = nchunk_of(cfg->V);
  const size_t cnt_bytes = align256(sizeof(unsigned int) * (size_t)(rows + cfg->B));
  const size_t need = cnt_bytes + sizeof(float) * (size_t)rows * nchunk * (2 + 2 * cfg->topk);
  ET_RETURN_IF(need > kExpandScratchBytes, ET_ERR_WORKSPACE);  // beyond the static scratch
  ET_RETURN_IF(!table_ptr(logits, &logits), ET_ERR_INVALID_ARG);  // device, or page-locked host memory
  void *scratch = nullptr;
  const et_status s = expand_scratch(&scratch);
  if (s != ET_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  // counters must start at zero; clear them on the caller's stream (no allocation)
  if (cudaMemsetAsync(scratch, 0, cnt_bytes, st) != cudaSuccess) return ET_ERR_CUDA;
  ExpandArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.row_of_node = row_of_node;
  a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
  a.B = cfg->B; a.V = cfg->V; a.k = cfg->topk; a.m = cfg->m; a.C = g.C; a.layer = layer; a.m_l = m_l;
  a.base_next = g.base[layer + 1];
  a.m_next = (layer + 1 < cfg->depth) ? g.expanded[layer + 1] : 0;
  a.nchunk = nchunk;
  a.tree = *tree;
  a.dev_status = dev_status;
  unsigned char *base = static_cast<unsigned char *>(scratch);
  a.row_cnt = reinterpret_cast<unsigned int *>(base);
  a.seq_cnt = a.row_cnt + rows;
  a.part = reinterpret_cast<float *>(base + cnt_bytes);
  if (cfg->V <= kClMaxV) return launch_expand_row(a, st);
  dim3 grid(a.nchunk, rows);
  const size_t smem = (size_t)a.nchunk * a.k * (sizeof(float) + sizeof(int));
  return et_launch(k_expand, grid, dim3(kExpThreads), smem, st, 0, a);
}
