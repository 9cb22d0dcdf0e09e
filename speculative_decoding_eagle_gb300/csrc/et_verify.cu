// Lossless acceptance walk on sm_103a (EAGLE blog "大模型系列——论文解读：
// eagle/eagle2", sections 1.1 and 1.2: one target pass verifies the whole
// draft and the output distribution is unchanged, greedy or not).
//
// Phase 1 (all blocks): every flat row's target logits are streamed once with
// 128-bit loads, split over blocks; each block reduces its slice (argmax, or
// max and sum of exp at temperature T) and the row's blocks merge them.  In
// the draft-q mode a row with children also decides its own acceptance there
// (p and q of the row, one cluster reduction per rejected child).
// Phase 2 (the last row-block of a sequence): walk the tree from the root,
// then draw the bonus token by an inverse CDF over the stopping row.
#include "et_common.cuh"
#include "et_cdf.cuh"

extern "C" __attribute__((visibility("hidden"))) int et_internal_table_ptr(const void *p, const void **dev);
extern "C" __attribute__((visibility("hidden"))) size_t et_internal_tree_ws(const et_tree_cfg *cfg, size_t *cnt_bytes, size_t *part_off,
                                      size_t *rowstat_off, size_t *dq_off);

namespace et {

constexpr int kVThreads = 256;
constexpr int kVVec = 2;
constexpr int kVChunk = kVThreads * 4 * kVVec;

struct VerifyArgs {
  int mode;
  int B, V, N, C, D, nchunk;
  float T;
  const float *tlog;
  long long tstride;
  const int32_t *tmap;
  const float *dlog;
  long long dstride;
  const int32_t *dmap;
  const float *uniforms;
  const int32_t *flat_node, *flat_tok, *flat_parent;
  int32_t *accept_len, *path, *tokens, *dev_status;
  float *part;        // [B*N][nchunk][2]
  float *rowstat;     // [B*N][2]
  float *dq;          // [B*N][8] per flat row: [3] the accepted child (int bits: row, -1 leaf, -2 all
                      // rejected), both stochastic modes; draft-q also [0..2]: q's max and sum, the residual's
                      // c once every child is rejected
  unsigned int *row_cnt, *seq_cnt;
  int vec4t, vec4d;       // 16-byte aligned target / draft rows
  int cdf_span, cdf_nch;  // chunk statistics of each row in part: span tokens each, nch chunks
};

__device__ __forceinline__ const float *table_row(const float *tab, long long stride, const int32_t *map, int C,
                                                  int b, int node, long long flat_row, int &bad) {
  long long r;
  if (map) {
    if (node < -1 || node >= C) { bad = 1; return nullptr; }
    r = map[(long long)b * (C + 1) + node + 1];
  } else {
    r = flat_row;
  }
  if (r < 0) { bad = 1; return nullptr; }
  return tab + r * stride;
}

// ---- draft-q acceptance: the residual after each rejection at a row ----
// p = softmax(z/T) and q = softmax(zd/T) at the row; r starts as p and each
// rejected child sets r <- max(r - q, 0) / Z, Z its sum (r is kept when
// Z = 0).  By induction r = max(p - c q, 0) / F with F = sum max(p - c q, 0):
// (c, F) = (0, 1) at first, and a rejection moves to c' = c + F, F' = F(c')
// (when F' > 0), because max(max(p - c q, 0) / F - q, 0) = max(p - c' q, 0) / F.
// The pairs depend on the row and on how many children were rejected, not on
// which tokens they were, and a child's test needs only p and q at its token,
// so phase 1 decides every row's acceptance in parallel (stopping at the first
// accepted child) and the walk follows the accepted children.
__device__ __forceinline__ float dq_weight(float y, float M, float inv_sum) {
  return y > -INFINITY ? exp_fast(y - M) * inv_sum : 0.f;
}
__device__ __forceinline__ float dq_excess(float p, float q, float c) { return fmaxf(fmaf(-c, q, p), 0.f); }

// ---- point-mass acceptance: every row decided in phase 1 ----
// A deterministic child x is a point-mass proposal, so its test is
// u < r(x) / sum(r) with r = p minus the tokens of the siblings rejected
// before it.  With e_i = exp(z(x_i) / T) (up to a common factor) for each
// distinct child token and S_rest the row's weight outside every child
// token, child k's ratio is e_k / (S_rest + sum_{i>=k} e_i): sums of positive
// terms only, so nothing cancels when the rejected siblings hold almost all
// of the mass.  The suffix sums run from the last child to the first as
// (max raw logit, sum of exp((z - max) / T)) pairs merged like a log-sum-exp,
// so each ratio is formed relative to its own largest term.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2, float invT) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) { m = M; s = 0.f; return; }
  s = (m > -INFINITY ? s * expf((m - M) * invT) : 0.f) + (m2 > -INFINITY ? s2 * expf((m2 - M) * invT) : 0.f);
  m = M;
}

// One warp decides a row with nkid > 0 children: kid[k] their flat rows in
// ascending order, zk[k] the raw target logit of each child's token at this
// row (-inf when the token is outside [0, V) or an earlier sibling holds it:
// no residual mass), uk[k] their uniforms, (Mr, Sr) the row's tokens outside
// the children.  Returns the first accepted child's flat row, or -2.
__device__ int pm_decide(int nkid, const int *kid, const float *zk, const float *uk, float Mr, float Sr, float invT) {
  const int lane = threadIdx.x & 31;
  float cm = Mr, cs = Sr;  // the rest plus every child after the current group
  int acc = -2;
  for (int g0 = ((nkid - 1) >> 5) << 5; g0 >= 0; g0 -= 32) {
    const int k = g0 + lane;
    const float z = k < nkid ? zk[k] : -INFINITY;
    float m = z, sm = z > -INFINITY ? 1.f : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // suffix merge inside the group: lane gets children k .. g0 + 31
      const float m2 = __shfl_down_sync(0xffffffffu, m, o), s2 = __shfl_down_sync(0xffffffffu, sm, o);
      if (lane + o < 32) lse_merge(m, sm, m2, s2, invT);
    }
    lse_merge(m, sm, cm, cs, invT);
    const float ratio = (z > -INFINITY && sm > 0.f) ? expf((z - m) * invT) / sm : 0.f;
    const unsigned int hit = __ballot_sync(0xffffffffu, k < nkid && uk[k] < ratio);
    if (hit) acc = kid[g0 + __ffs(hit) - 1];  // groups run last to first: the earliest hit wins
    cm = __shfl_sync(0xffffffffu, m, 0);
    cs = __shfl_sync(0xffffffffu, sm, 0);
  }
  return acc;
}

// The tokens, raw target logits and uniforms of a row's children (by child
// rank) into shared memory, by the block's threads; a token already held by
// an earlier sibling, or outside [0, V), gets logit -inf.  The caller
// synchronises before reading them.
__device__ void pm_child_inputs(const VerifyArgs &a, long long fo, const int *kid, int nkid, const float *zrow,
                                int *ktok, float *zk, float *uk) {
  for (int k = threadIdx.x; k < nkid; k += blockDim.x) ktok[k] = a.flat_tok[fo + kid[k]];
  __syncthreads();
  for (int k = threadIdx.x; k < nkid; k += blockDim.x) {
    const int x = ktok[k];
    bool ok = zrow && x >= 0 && x < a.V;
    for (int i = 0; i < k && ok; ++i) ok = ktok[i] != x;
    int f2 = 0;
    zk[k] = ok ? sanitize_logit(__ldg(zrow + x), f2) : -INFINITY;
    uk[k] = a.uniforms[fo + kid[k]];
  }
}

// Bitmap of the children's tokens inside [lo, lo + 32 * words) (point-mass
// rows: their chunk sums leave those tokens out).  Every thread calls it; the
// bitmap must be zero on entry.
__device__ __forceinline__ void mark_child_tokens(const VerifyArgs &a, long long fo, const int *kid, int nkid, int lo,
                                                  int words, unsigned int *bits) {
  for (int k = threadIdx.x; k < nkid; k += blockDim.x) {
    const int off = a.flat_tok[fo + kid[k]] - lo;
    if (off >= 0 && off < 32 * words) atomicOr(&bits[off >> 5], 1u << (off & 31));
  }
  __syncthreads();
}

// Draft-q test of one child from p and q at its token and the residual
// (c, F) in force: u < min(1, r(x) / q(x)).  Phase 1 evaluates it identically
// in every block of a row's cluster.
__device__ __forceinline__ bool dq_accept(float zt, float zd, bool ok, float u, float invT, float M, float invS,
                                          float Mq, float invSq, float c, float F) {
  const float qx = dq_weight(__fmul_rn(zd, invT), Mq, invSq);
  const float px = dq_weight(__fmul_rn(zt, invT), M, invS);
  const float r = F > 0.f ? dq_excess(px, qx, c) / F : 0.f;
  const float ratio = qx <= 0.f ? 1.f : fminf(1.f, r / qx);
  return ok && u < ratio;
}

// The children of row i (rows after i whose parent is i), in row order, by
// warp 0; every thread gets the count.  parents = the sequence's flat_parent.
template <int NT>
__device__ int child_list(const int32_t *parents, int N, int i, int *list, int *count) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = 0;
    for (int j0 = i + 1; j0 < N; j0 += 32) {
      const int j = j0 + lane;
      const bool c = j < N && parents[j] == i;
      const unsigned int m = __ballot_sync(0xffffffffu, c);
      if (c) list[n + __popc(m & ((1u << lane) - 1u))] = j;
      n += __popc(m);
    }
    if (lane == 0) *count = n;
  }
  __syncthreads();
  return *count;
}

struct WalkSmem {
  float redz[32];
  int redi[32];
  float cdf_tsum[kMaxV / kVChunk];  // per chunk weights of the bonus draw
  int par[kMaxN], tokf[kMaxN], nodef[kMaxN];
  float rs0[kMaxN], rs1[kMaxN];  // per flat row: argmax id (bits) / max, -, / sum
  float qs0[kMaxN], qs1[kMaxN];  // draft-q: max and sum of q at each row
  float zc[kMaxN];               // phase 1: target logit of each child's token (by child rank)
  float dc[kMaxN];               // phase 1, draft-q: draft logit of each child's token (by child rank)
  int ktok[kMaxN];               // phase 1, point-mass: each child's token (by child rank)
  float cf[kMaxN];               // draft-q: c of the residual once all of a row's children are rejected
  int acc[kMaxN];                // accepted child of each row (-1 leaf, -2 all rejected)
  int kid[kMaxN];                // phase 1: the children of the block's row
  int opath[kMaxDepth + 2], otok[kMaxDepth + 2];
  int rej[kMaxN];                // the tokens of the stop row's children (all rejected)
  unsigned int rejbits[kMaxSpanWords];  // phase 1: children's tokens in the block's span; bonus draw: rejected
                                        // children inside the chunk being scanned
  float s_M, s_S;
  float uni[kMaxN];      // this sequence's uniforms
  int s_nrej, s_cur, s_alen, s_kids, s_nkid;
};

// Phase 2 of acceptance, run by the last row-block of sequence b: everything
// the walk needs (row statistics, the decision phase 1 took at each row,
// uniforms) is fetched in parallel; greedy: every row's accepted child (its
// first child whose token is the row's argmax) is found at once by shared-
// memory atomics; one warp then walks the accepted children from the root
// (stochastic: the child phase 1 accepted at each row); the block draws the
// bonus token at the row where the walk stops.
template <int NT, bool kDraftQ>
__device__ void verify_walk(const VerifyArgs &a, int b, WalkSmem &w) {
  const int t = threadIdx.x;
  int *par = w.par, *tokf = w.tokf, *nodef = w.nodef, *rej = w.rej;
  const int N = a.N;
  const long long fo = (long long)b * N;
  const bool greedy = a.mode == ET_ACCEPT_GREEDY, dq = kDraftQ && a.mode == ET_ACCEPT_STOCH_DRAFTQ;
  const float invT = 1.f / a.T;
  const auto child_of = [&](int ac, int j) { return (ac > j && ac < N) || ac == -2 ? ac : -1; };
  int badp = 0;
  for (int j = t; j < N; j += NT) {
    const int p = a.flat_parent[fo + j], x = a.flat_tok[fo + j];
    par[j] = p;
    tokf[j] = x;
    nodef[j] = a.flat_node[fo + j];
    w.rs0[j] = ld_cg(a.rowstat + 2 * (fo + j));
    w.rs1[j] = ld_cg(a.rowstat + 2 * (fo + j) + 1);
    if (!greedy) w.uni[j] = a.uniforms[fo + j];
    if (dq) {  // the row's record, written in phase 1
      const float4 lo4 = ld_cg(reinterpret_cast<const float4 *>(a.dq) + 2 * (fo + j));
      w.qs0[j] = lo4.x;
      w.qs1[j] = lo4.y;
      w.cf[j] = lo4.z;
      w.acc[j] = child_of(__float_as_int(lo4.w), j);
    } else if (!greedy) {  // point-mass: the decision phase 1 took at the row
      w.acc[j] = child_of(__float_as_int(ld_cg(a.dq + 8 * (fo + j) + 3)), j);
    } else {
      w.acc[j] = 0x7fffffff;  // greedy: filled below
    }
  }
  __syncthreads();
  if (greedy) {  // every row's accepted child at once: its first child carrying the row's argmax token
    for (int j = t; j < N; j += NT) {
      const int p = par[j];
      if (p >= 0 && p < j && tokf[j] == __float_as_int(w.rs0[p])) atomicMin(&w.acc[p], j);
    }
    __syncthreads();
  }
  if (t < 32) {  // one warp walks the accepted children
    const int lane = t;
    int cur = 0, alen = 0, nrej = 0, kids = 0;
    if (lane == 0) w.opath[0] = 0;
    for (int iter = 0; iter <= a.D; ++iter) {
      int nxt = -1;
      nrej = 0;
      kids = 0;
      if (greedy) {
        const int am = __float_as_int(w.rs0[cur]);
        const int ac = w.acc[cur];  // the first row (ascending) that is a child with token am
        nxt = ac < N ? ac : -1;
        if (nxt < 0 && lane == 0) w.otok[alen] = am;
      } else {  // stochastic: phase 1 decided every row
        const int ac = w.acc[cur];
        nxt = ac >= 0 ? ac : -1;
        kids = ac == -2;
      }
      if (nxt < 0 || alen >= a.D) break;
      if (lane == 0) {
        w.otok[alen] = tokf[nxt];
        w.opath[alen + 1] = nxt;
      }
      ++alen;
      cur = nxt;
    }
    if (!greedy && !dq && kids) {  // point-mass, every child rejected: the draw leaves out their tokens
      for (int j0 = cur + 1; j0 < N; j0 += 32) {
        const int j = j0 + lane;
        const bool c = j < N && par[j] == cur;
        const unsigned int m = __ballot_sync(0xffffffffu, c);
        if (c) rej[nrej + __popc(m & ((1u << lane) - 1u))] = tokf[j];
        nrej += __popc(m);
      }
    }
    if (lane == 0) {
      w.s_cur = cur;
      w.s_nrej = nrej;
      w.s_alen = alen;
      w.s_kids = kids;
    }
  }
  __syncthreads();
  const int alen = w.s_alen;
  if (!greedy) {  // bonus token: inverse CDF of the residual at the stop row
    const int cur = w.s_cur;
    int badz = 0;
    const float *zr = table_row(a.tlog, a.tstride, a.tmap, a.C, b, nodef[cur], fo + cur, badz);
    const float *cst = a.part + (fo + cur) * (long long)a.nchunk * 2;
    const CdfRow cdf{a.cdf_span, a.cdf_nch, a.V, a.vec4t, a.T, invT};  // chunk maxima are raw logits
    int bonus;
    if (dq && w.s_kids > 0) {  // every child rejected: phase 1 left the chunk sums of max(p - c q, 0)
      const float *dr = table_row(a.dlog, a.dstride, a.dmap, a.C, b, nodef[cur], fo + cur, badz);
      const float M = w.rs0[cur], S = w.rs1[cur], Mq = w.qs0[cur], Sq = w.qs1[cur], c = w.cf[cur];
      const float invS = S > 0.f ? 1.f / S : 0.f, invSq = Sq > 0.f ? 1.f / Sq : 0.f;
      bonus = chunk_inverse_cdf<NT, true>(cdf, zr, dr, a.vec4d, cst, M, w.uni[0], nullptr, 0, w.redz, w.redi,
                                          w.cdf_tsum, w.rejbits, [&](float zt, float zd) -> float {
                                            return dq_excess(dq_weight(__fmul_rn(zt, invT), M, invS),
                                                             dq_weight(__fmul_rn(zd, invT), Mq, invSq), c);
                                          });
    } else {  // point-mass residual (the children's tokens already out of the chunk sums), or a leaf: p
      bonus = bonus_from_chunks<NT, true>(cdf, zr, cst, w.rs0[cur], w.uni[0], rej, w.s_nrej, w.redz, w.redi,
                                          w.cdf_tsum, w.rejbits);
    }
    if (t == 0) w.otok[alen] = bonus;
    badp |= badz;
  }
  __syncthreads();
  const long long po = (long long)b * (a.D + 1);
  for (int j = t; j <= a.D; j += NT) {
    a.path[po + j] = j <= alen ? w.opath[j] : -1;
    a.tokens[po + j] = j <= alen ? w.otok[j] : -1;
  }
  if (t == 0) a.accept_len[b] = alen;
  if (badp) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
}

// Draft-q phase 1 of one row, by one block (rows too long for one cluster):
// q's max and sum, then the children in row order, each tested against the
// residual in force and, when rejected, one pass over the row for the next
// (c, F); when every child is rejected, the chunk sums of max(p - c q, 0) for
// the bonus draw.  Returns whether the row has children.
template <int NT>
__device__ bool dq_row_block(const VerifyArgs &a, long long row, int b, int node, const float *zr, float M, float S,
                             WalkSmem &w) {
  const int t = threadIdx.x;
  const int i = (int)(row - (long long)b * a.N);
  const long long fo = row - i;
  const int nkid = child_list<NT>(a.flat_parent + fo, a.N, i, w.kid, &w.s_nkid);
  if (nkid == 0) {
    if (t == 0) a.dq[8 * row + 3] = __int_as_float(-1);  // a leaf
    return false;
  }
  int bad = 0, flag = 0;
  const float *dr = table_row(a.dlog, a.dstride, a.dmap, a.C, b, node, row, bad);
  const float invT = 1.f / a.T, invS = S > 0.f ? 1.f / S : 0.f;
  for (int k = t; k < nkid; k += NT) {
    const long long j = fo + w.kid[k];
    const int x = a.flat_tok[j];
    const bool ok = x >= 0 && x < a.V;
    int f2 = 0;
    w.zc[k] = (ok && zr) ? sanitize_logit(zr[x], f2) : -INFINITY;
    w.dc[k] = (ok && dr) ? sanitize_logit(dr[x], f2) : -INFINITY;
    w.uni[k] = a.uniforms[j];
    w.tokf[k] = ok;
    if (!ok) bad = 1;
  }
  auto yd = [&](int v) -> float { return dr ? __fmul_rn(sanitize_logit(dr[v], flag), invT) : -INFINITY; };
  auto yt = [&](int v) -> float { return zr ? __fmul_rn(sanitize_logit(zr[v], flag), invT) : -INFINITY; };
  float lq = -INFINITY;
  for (int v = t; v < a.V; v += NT) lq = fmaxf(lq, yd(v));
  const float Mq = block_max<NT>(lq, w.redz);  // its barriers publish the children's values above
  float ls = 0.f;
  if (Mq > -INFINITY)
    for (int v = t; v < a.V; v += NT) ls += exp_fast(yd(v) - Mq);
  const float Sq = block_sum<NT>(ls, w.redz);
  const float invSq = Sq > 0.f ? 1.f / Sq : 0.f;
  float c = 0.f, F = 1.f;
  int acc = -2;
  for (int k = 0; k < nkid; ++k) {
    if (dq_accept(w.zc[k], w.dc[k], w.tokf[k] != 0, w.uni[k], invT, M, invS, Mq, invSq, c, F)) {
      acc = w.kid[k];
      break;
    }
    const float c1 = c + F;
    float loc = 0.f;
    for (int v = t; v < a.V; v += NT) loc += dq_excess(dq_weight(yt(v), M, invS), dq_weight(yd(v), Mq, invSq), c1);
    const float F1 = block_sum<NT>(loc, w.redz);
    if (F1 > 0.f) { c = c1; F = F1; }
  }
  if (t == 0) {
    a.dq[8 * row] = Mq;
    a.dq[8 * row + 1] = Sq;
    a.dq[8 * row + 2] = c;
    a.dq[8 * row + 3] = __int_as_float(acc);
  }
  if (acc < 0) {
    float *cst = a.part + row * a.nchunk * 2;
    for (int ch = 0; ch < a.nchunk; ++ch) {
      float loc = 0.f;
      for (int e = t; e < kVChunk; e += NT) {
        const int v = ch * kVChunk + e;
        if (v < a.V) loc += dq_excess(dq_weight(yt(v), M, invS), dq_weight(yd(v), Mq, invSq), c);
      }
      const float sum = block_sum<NT>(loc, w.redz);
      if (t == 0) { cst[2 * ch] = M; cst[2 * ch + 1] = sum; }
    }
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  return true;
}

__global__ void __launch_bounds__(kVThreads) k_verify(VerifyArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  __shared__ WalkSmem w;
  __shared__ int sflag;
  float *redz = w.redz;
  int *redi = w.redi;

  const int t = threadIdx.x;
  const int row = blockIdx.y, c = blockIdx.x;
  const int b = row / a.N;
  int flag = 0, bad = 0;
  const int node = a.flat_node[row];
  const float *zrow = table_row(a.tlog, a.tstride, a.tmap, a.C, b, node, row, bad);

  float v[4 * kVVec];
  const int c0 = c * kVChunk;
#pragma unroll
  for (int u = 0; u < kVVec; ++u) {
    const int e0 = c0 + (u * kVThreads + t) * 4;
    if (zrow && a.vec4t && e0 + 3 < a.V) {
      float4 f = __ldg(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u + 0] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < a.V) ? __ldg(zrow + e0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (e0 + j < a.V) v[4 * u + j] = sanitize_logit(v[4 * u + j], flag);
  }
  const int i = row - b * a.N;
  const long long fo = (long long)row - i;
  int nkid = 0;
  if (a.mode == ET_ACCEPT_STOCH_POINT) {  // the chunk's sums leave out the tokens of the row's children
    constexpr int kWords = kVChunk / 32;
    for (int x = t; x < kWords; x += kVThreads) w.rejbits[x] = 0u;
    nkid = child_list<kVThreads>(a.flat_parent + fo, a.N, i, w.kid, &w.s_nkid);
    if (nkid > 0) {
      mark_child_tokens(a, fo, w.kid, nkid, c0, kWords, w.rejbits);
#pragma unroll
      for (int j = 0; j < 4 * kVVec; ++j) {
        const int off = ((j >> 2) * kVThreads + t) * 4 + (j & 3);
        if ((w.rejbits[off >> 5] >> (off & 31)) & 1u) v[j] = -INFINITY;
      }
    }
  }
  float *prt = a.part + ((long long)row * a.nchunk + c) * 2;
  if (a.mode == ET_ACCEPT_GREEDY) {
    float bz = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 4 * kVVec; ++j) {
      const int e = c0 + ((j >> 2) * kVThreads + t) * 4 + (j & 3);
      if (e < a.V && ranks_before(v[j], e, bz, bi)) { bz = v[j]; bi = e; }
    }
    block_best<kVThreads>(bz, bi, redz, redi);
    if (t == 0) { prt[0] = bz; prt[1] = __int_as_float(bi); }
  } else {  // (max of the raw logits, sum of exp((z - max) / T)) of the chunk
    const float invT = 1.f / a.T;
    float lm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4 * kVVec; ++j) lm = fmaxf(lm, v[j]);
    const float Mc = block_max<kVThreads>(lm, redz);
    float ls = 0.f;
    if (Mc > -INFINITY) {
#pragma unroll
      for (int j = 0; j < 4 * kVVec; ++j) ls += v[j] > -INFINITY ? expf((v[j] - Mc) * invT) : 0.f;
    }
    const float Sc = block_sum<kVThreads>(ls, redz);
    if (t == 0) { prt[0] = Mc; prt[1] = Sc; }
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && c == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);

  if (!arrive_last(&a.row_cnt[row], (unsigned)a.nchunk, &sflag)) return;
  {
    const float *rp = a.part + (long long)row * a.nchunk * 2;
    if (a.mode == ET_ACCEPT_GREEDY) {
      float bz = -INFINITY;
      int bi = 0x7fffffff;
      for (int cc = t; cc < a.nchunk; cc += kVThreads) {
        const float z = ld_cg(rp + 2 * cc);
        const int id = __float_as_int(ld_cg(rp + 2 * cc + 1));
        if (ranks_before(z, id, bz, bi)) { bz = z; bi = id; }
      }
      block_best<kVThreads>(bz, bi, redz, redi);
      if (t == 0) { a.rowstat[2 * row] = __int_as_float(bi); a.rowstat[2 * row + 1] = bz; }
    } else {
      const float invT = 1.f / a.T;
      float cm = -INFINITY, cs = 0.f;
      if (t < a.nchunk) { cm = ld_cg(rp + 2 * t); cs = ld_cg(rp + 2 * t + 1); }
      const float M = block_max<kVThreads>(cm, redz);
      const float S =
          block_sum<kVThreads>((t < a.nchunk && cm > -INFINITY) ? cs * expf((cm - M) * invT) : 0.f, redz);
      if (a.mode == ET_ACCEPT_STOCH_DRAFTQ) {
        // the residual arithmetic runs on z / T: its maximum is fl(M / T), the sum is the same
        const bool kids = dq_row_block<kVThreads>(a, row, b, node, zrow, __fmul_rn(M, invT), S, w);
        if (t == 0) { a.rowstat[2 * row] = kids ? __fmul_rn(M, invT) : M; a.rowstat[2 * row + 1] = S; }
      } else {
        if (t == 0) { a.rowstat[2 * row] = M; a.rowstat[2 * row + 1] = S; }
        int acc = -1;  // a leaf
        if (nkid > 0) {
          pm_child_inputs(a, fo, w.kid, nkid, zrow, w.ktok, w.zc, w.uni);
          __syncthreads();
          if (t < 32) acc = pm_decide(nkid, w.kid, w.zc, w.uni, M, S, invT);
        }
        if (t == 0) a.dq[8 * (long long)row + 3] = __int_as_float(acc);
      }
    }
  }
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.N, &sflag)) return;

  verify_walk<kVThreads, true>(a, b, w);
}

// ---------------------------------------------------------------------------
// phase 1 on a thread-block cluster per flat row (V <= 32768): CTA q reduces
// logits [4096 q, 4096 q + 4096) and stores its result straight into the
// leader's shared memory; after one cluster barrier the leader merges them
// and writes the row's statistic.  A draft-q row with children also keeps its
// slice of p and q in registers and runs one cluster reduction per child for
// the residual sums.
// ---------------------------------------------------------------------------
constexpr int kVClThreads = 256;
constexpr int kVClVec = 4;
constexpr int kVClSpan = kVClThreads * 4 * kVClVec;
constexpr int kVClMaxCtas = 8;
constexpr int kVClMaxV = kVClSpan * kVClMaxCtas;

// this block's slice of a row, sanitised; -inf past the end or without a row
__device__ __forceinline__ void cl_load_span(const float *row, int base, int vec4, int V, float (&v)[4 * kVClVec],
                                             int &flag) {
  const int t = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kVClVec; ++u) {
    const int e0 = base + u * kVClThreads * 4 + t * 4;
    if (row && vec4 && e0 + 3 < V) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(row + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (row && e0 + j < V) ? __ldg(row + e0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (e0 + j < V) v[4 * u + j] = sanitize_logit(v[4 * u + j], flag);
  }
}

// kDraftQ: the draft-q instance (rows with children take the residual branch);
// the other modes use an instance without it and its registers.
template <bool kDraftQ>
__global__ void __launch_bounds__(kVClThreads) k_verify_cl(VerifyArgs a) {
  constexpr int NW = kVClThreads / 32;
  __shared__ WalkSmem w;
  __shared__ unsigned long long wkey[NW], gkey[kVClMaxCtas];
  __shared__ float wmax[NW], wsum[NW], wmaxq[NW], wsumq[NW];
  __shared__ float2 gms[kVClMaxCtas];
  __shared__ float4 g4[kVClMaxCtas];            // draft-q: (max, sum) of p and of q, per block
  __shared__ float zpart[2][kVClMaxCtas * NW];  // draft-q: per-warp residual sums, alternating buffers
  __shared__ int sflag;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int R = gridDim.x;
  const int q = (int)cl_rank();
  const int row = blockIdx.y;
  const int b = row / a.N, i = row - b * a.N;
  cl_arrive_relaxed();  // phase 0: this block has started (waited on before any remote store)
  pdl_wait();           // the previous kernel in the stream has completed
  pdl_trigger();        // only now may the next kernel launch: at most one waits ahead
  int flag = 0, bad = 0;
  const int node = a.flat_node[row];
  const float *zrow = table_row(a.tlog, a.tstride, a.tmap, a.C, b, node, row, bad);
  const int base = q * kVClSpan;
  float v[4 * kVClVec];
  cl_load_span(zrow, base, a.vec4t, a.V, v, flag);
  const bool greedy = a.mode == ET_ACCEPT_GREEDY;
  const long long fo = (long long)row - i;
  int nkid = 0;
  if (!greedy) {  // the children of this row (every block of the cluster finds the same)
    if (!kDraftQ)
      for (int x = t; x < kVClSpan / 32; x += kVClThreads) w.rejbits[x] = 0u;
    nkid = child_list<kVClThreads>(a.flat_parent + fo, a.N, i, w.kid, &w.s_nkid);
  }
  if (!kDraftQ && nkid > 0) {
    // point-mass: this block's sums leave out the children's tokens, and the
    // leader fetches the children's logits for the row's decision
    mark_child_tokens(a, fo, w.kid, nkid, base, kVClSpan / 32, w.rejbits);
#pragma unroll
    for (int e = 0; e < 4 * kVClVec; ++e) {
      const int off = (e >> 2) * (kVClThreads * 4) + t * 4 + (e & 3);
      if ((w.rejbits[off >> 5] >> (off & 31)) & 1u) v[e] = -INFINITY;
    }
    if (q == 0) pm_child_inputs(a, fo, w.kid, nkid, zrow, w.ktok, w.zc, w.uni);
  }
  if (kDraftQ && nkid > 0) {
    const float invT = 1.f / a.T;
    const float *drow = table_row(a.dlog, a.dstride, a.dmap, a.C, b, node, row, bad);
    // every block loads each child's token logits and uniform: the tests below
    // are evaluated alike in all blocks of the cluster
    for (int k = t; k < nkid; k += kVClThreads) {
      const long long j = fo + w.kid[k];
      const int x = a.flat_tok[j];
      const bool ok = x >= 0 && x < a.V;
      int f2 = 0;
      w.zc[k] = (ok && zrow) ? sanitize_logit(__ldg(zrow + x), f2) : -INFINITY;
      w.dc[k] = (ok && drow) ? sanitize_logit(__ldg(drow + x), f2) : -INFINITY;
      w.uni[k] = a.uniforms[j];
      w.tokf[k] = ok;
      if (!ok && q == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    }
    float d[4 * kVClVec];
    cl_load_span(drow, base, a.vec4d, a.V, d, flag);
    float lm = -INFINITY, lq = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4 * kVClVec; ++e) {
      v[e] = __fmul_rn(v[e], invT);
      d[e] = __fmul_rn(d[e], invT);
      lm = fmaxf(lm, v[e]);
      lq = fmaxf(lq, d[e]);
    }
    lm = warp_max(lm);
    lq = warp_max(lq);
    if (lane == 0) { wmax[warp] = lm; wmaxq[warp] = lq; }
    if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
    if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    __syncthreads();
    cl_wait();  // phase 0 done: every block of the cluster runs
    float Mc = -INFINITY, Mqc = -INFINITY;
#pragma unroll
    for (int x = 0; x < NW; ++x) { Mc = fmaxf(Mc, wmax[x]); Mqc = fmaxf(Mqc, wmaxq[x]); }
    float ls = 0.f, lsq = 0.f;
#pragma unroll
    for (int e = 0; e < 4 * kVClVec; ++e) {
      if (Mc > -INFINITY) ls += exp_fast(v[e] - Mc);
      if (Mqc > -INFINITY) lsq += exp_fast(d[e] - Mqc);
    }
    ls = warp_sum(ls);
    lsq = warp_sum(lsq);
    if (lane == 0) { wsum[warp] = ls; wsumq[warp] = lsq; }
    __syncthreads();
    if (t == 0) {  // every block gets every block's statistics
      float Sc = 0.f, Sqc = 0.f;
#pragma unroll
      for (int x = 0; x < NW; ++x) { Sc += wsum[x]; Sqc += wsumq[x]; }
      for (int x = 0; x < R; ++x) cl_st_f32x4(cl_map(&g4[q], x), Mc, Sc, Mqc, Sqc);
    }
    cl_arrive();
    cl_wait();
    float M = -INFINITY, Mq = -INFINITY, S = 0.f, Sq = 0.f;
    for (int x = 0; x < R; ++x) { M = fmaxf(M, g4[x].x); Mq = fmaxf(Mq, g4[x].z); }
    for (int x = 0; x < R; ++x) {  // the same order in every block: the same M, S, Mq, Sq
      const float4 g = g4[x];
      S += g.x > -INFINITY ? g.y * expf(g.x - M) : 0.f;
      Sq += g.z > -INFINITY ? g.w * expf(g.z - Mq) : 0.f;
    }
    const float invS = S > 0.f ? 1.f / S : 0.f, invSq = Sq > 0.f ? 1.f / Sq : 0.f;
#pragma unroll
    for (int e = 0; e < 4 * kVClVec; ++e) {
      v[e] = dq_weight(v[e], M, invS);    // p
      d[e] = dq_weight(d[e], Mq, invSq);  // q
    }
    float c = 0.f, F = 1.f;  // the residual in force: max(p - c q, 0) / F
    int acc = -2;
    for (int k = 0; k < nkid; ++k) {  // each child in row order; a rejection moves the residual on
      if (dq_accept(w.zc[k], w.dc[k], w.tokf[k] != 0, w.uni[k], invT, M, invS, Mq, invSq, c, F)) {
        acc = w.kid[k];
        break;
      }
      const float c1 = c + F;
      float loc = 0.f;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) loc += dq_excess(v[e], d[e], c1);
      loc = warp_sum(loc);
      // every warp's sum into every block; a buffer is rewritten two children
      // later, after every block has passed the barrier in between
      if (lane < R) cl_st_f32(cl_map(&zpart[k & 1][q * NW + warp], lane), loc);
      cl_arrive();
      cl_wait();
      const int ns = R * NW;  // <= 64: two per lane, then the same butterfly in every warp
      float z = (lane < ns ? zpart[k & 1][lane] : 0.f) + (lane + 32 < ns ? zpart[k & 1][lane + 32] : 0.f);
      z = warp_sum(z);
      if (z > 0.f) { c = c1; F = z; }
    }
    if (q == 0 && t == 0) {
      a.rowstat[2 * row] = M;
      a.rowstat[2 * row + 1] = S;
      a.dq[8 * (long long)row] = Mq;
      a.dq[8 * (long long)row + 1] = Sq;
      a.dq[8 * (long long)row + 2] = c;
      a.dq[8 * (long long)row + 3] = __int_as_float(acc);
    }
    if (acc >= 0) {  // a child is accepted: the walk never draws a bonus token here
      if (q != 0) return;
    } else {  // every child rejected: the chunk sums of max(p - c q, 0) for the bonus draw
      float loc = 0.f;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) loc += dq_excess(v[e], d[e], c);
      loc = warp_sum(loc);
      if (lane == 0) wsum[warp] = loc;
      __syncthreads();
      if (t == 0) {  // this chunk's sum of max(p - c q, 0), to the leader
        float bs = 0.f;
#pragma unroll
        for (int x = 0; x < NW; ++x) bs += wsum[x];
        cl_st_f32x2(cl_map(&gms[q], 0), M, bs);
      }
      cl_arrive();
      if (q != 0) return;
      cl_wait();
      if (t == 0) {  // chunk weight = sum * exp(M - M): the plain sums
        float *cst = a.part + (long long)row * a.nchunk * 2;
        for (int x = 0; x < R; ++x) { cst[2 * x] = gms[x].x; cst[2 * x + 1] = gms[x].y; }
      }
    }
  } else {
    if (kDraftQ && q == 0 && t == 0) a.dq[8 * (long long)row + 3] = __int_as_float(-1);  // a leaf
    if (greedy) {  // (z desc, id asc) as one ascending key: the warp's best is its minimum
      unsigned long long best = ~0ull;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) {
        const int id = base + (e >> 2) * (kVClThreads * 4) + t * 4 + (e & 3);
        if (id < a.V) {
          const unsigned long long kk = zid_key(v[e], (unsigned int)id);
          best = kk < best ? kk : best;
        }
      }
      best = warp_min_u64(best);
      if (lane == 0) wkey[warp] = best;
    } else {  // (max of the raw logits, sum of exp((z - max) / T)) of this block's slice
      float lm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) lm = fmaxf(lm, v[e]);
      lm = warp_max(lm);
      if (lane == 0) wmax[warp] = lm;
    }
    if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
    if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    __syncthreads();
    cl_wait();  // phase 0 done: every block of the cluster runs
    if (greedy) {
      if (warp == 0) {
        const unsigned long long kk = warp_min_u64(wkey[lane & (NW - 1)]);
        if (lane == 0) cl_st_u64(cl_map(&gkey[q], 0), kk);
      }
    } else {
      const float invT = 1.f / a.T;
      float Mq = wmax[0];
#pragma unroll
      for (int x = 1; x < NW; ++x) Mq = fmaxf(Mq, wmax[x]);
      float ls = 0.f;
      if (Mq > -INFINITY) {
#pragma unroll
        for (int e = 0; e < 4 * kVClVec; ++e) ls += exp_fast((v[e] - Mq) * invT);
      }
      ls = warp_sum(ls);
      if (lane == 0) wsum[warp] = ls;
      __syncthreads();
      if (t == 0) {
        float Sq = 0.f;
#pragma unroll
        for (int x = 0; x < NW; ++x) Sq += wsum[x];
        cl_st_f32x2(cl_map(&gms[q], 0), Mq, Sq);
      }
    }
    cl_arrive();  // phase 1: release this block's stores
    if (q != 0) return;
    cl_wait();
    if (t == 0) {
      if (greedy) {
        unsigned long long kk = gkey[0];
        for (int x = 1; x < R; ++x) kk = gkey[x] < kk ? gkey[x] : kk;
        a.rowstat[2 * row] = __int_as_float((int)zid_id(kk));
        a.rowstat[2 * row + 1] = zid_value(kk);
      } else {
        const float invT = 1.f / a.T;
        float M = -INFINITY;
        for (int x = 0; x < R; ++x) M = fmaxf(M, gms[x].x);
        float S = 0.f;
        for (int x = 0; x < R; ++x) S += gms[x].x > -INFINITY ? gms[x].y * expf((gms[x].x - M) * invT) : 0.f;
        a.rowstat[2 * row] = M;
        a.rowstat[2 * row + 1] = S;
        float *cst = a.part + (long long)row * a.nchunk * 2;  // chunk statistics for the bonus draw
        for (int x = 0; x < R; ++x) { cst[2 * x] = gms[x].x; cst[2 * x + 1] = gms[x].y; }
        w.s_M = M;
        w.s_S = S;
      }
    }
    if (!kDraftQ && !greedy) {  // point-mass: the row's decision, by one warp
      __syncthreads();
      int acc = -1;  // a leaf
      if (nkid > 0 && t < 32) acc = pm_decide(nkid, w.kid, w.zc, w.uni, w.s_M, w.s_S, 1.f / a.T);
      if (t == 0) a.dq[8 * (long long)row + 3] = __int_as_float(acc);
    }
  }
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.N, &sflag)) return;
  verify_walk<kVClThreads, kDraftQ>(a, b, w);
}

// ---------------------------------------------------------------------------
// Acceptance as one walk per sequence (greedy and point-mass, V <= 32768),
// for batches large enough that reading every flat row costs more than the
// walk's dependent steps: one cluster of ceil(V / 4096) CTAs per sequence
// follows the accepted children from the root, reading only the rows on the
// path and the row it stops at (at most D + 1 of the N rows).  Each step is
// the parallel kernel's phase 1 for one row: every CTA reduces its 4096-token
// slice (greedy: the best (value desc, id asc) key; point-mass: (max raw
// logit, sum of exp((z - max) / T)) with the children's tokens left out),
// stores it into every CTA of the cluster (by step parity), and after one
// cluster barrier every CTA merges the slices in CTA order and decides the
// row the same way (greedy: the first child carrying the argmax token;
// point-mass: pm_decide on the same inputs), so the CTAs walk in step.  At
// the stop row the leader CTA draws the bonus token (greedy: the argmax;
// point-mass: the chunk inverse CDF of the residual, the slices' statistics
// being its chunks).
// ---------------------------------------------------------------------------
// From this many sequences on, greedy and point-mass acceptance walk each
// sequence's path in one cluster (measured on GB300 at the 7B shape,
// point-mass: 32 sequences 182 us reading every row against 25 us walking,
// 16 sequences 97 against 29 us; at batch 1 the parallel kernel's 8 us beats
// the walk's dependent steps).
constexpr int kSeqWalkMinB = 8;

struct SeqWalkSmem {
  int par[kMaxN], tok[kMaxN], node[kMaxN];
  int kid[kMaxN];
  int ktok[kMaxN];
  float zk[kMaxN], uk[kMaxN];
  unsigned int rejbits[kMaxSpanWords];
  unsigned long long wkey[kVClThreads / 32];
  float wmax[kVClThreads / 32], wsum[kVClThreads / 32];
  unsigned long long gkey[2][kVClMaxCtas];  // every CTA's best key, by step parity
  float2 gms[2][kVClMaxCtas];               // every CTA's (max, sum), by step parity
  int opath[kMaxDepth + 2], otok[kMaxDepth + 2];
  int rej[kMaxN];
  float redz[32];
  int redi[32];
  float cdf_tsum[kMaxV / kVChunk];
  int s_nkid, s_acc;
};

__global__ void __launch_bounds__(kVClThreads) k_verify_seq(VerifyArgs a) {
  constexpr int NW = kVClThreads / 32;
  __shared__ SeqWalkSmem w;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int R = gridDim.x;
  const int q = (int)cl_rank();
  const int b = blockIdx.y;
  const int N = a.N;
  const long long fo = (long long)b * N;
  const bool greedy = a.mode == ET_ACCEPT_GREEDY;
  const float invT = 1.f / a.T;
  cl_arrive_relaxed();  // this block has started (waited on before any remote store)
  pdl_wait();           // the previous kernel in the stream has completed
  pdl_trigger();        // only now may the next kernel launch: at most one waits ahead
  for (int j = t; j < N; j += kVClThreads) {
    w.par[j] = a.flat_parent[fo + j];
    w.tok[j] = a.flat_tok[fo + j];
    w.node[j] = a.flat_node[fo + j];
  }
  if (t == 0) w.opath[0] = 0;
  __syncthreads();
  cl_wait();
  const int base = q * kVClSpan;
  int cur = 0, alen = 0, flag = 0, badp = 0;
  float M = -INFINITY, S = 0.f;
  int am = -1, acc = -1, nkid = 0;
  const float *zrow = nullptr;
  for (int step = 0; step <= a.D; ++step) {
    const int par = step & 1;
    nkid = child_list<kVClThreads>(w.par, N, cur, w.kid, &w.s_nkid);
    int bad = 0;
    zrow = table_row(a.tlog, a.tstride, a.tmap, a.C, b, w.node[cur], fo + cur, bad);
    badp |= bad;
    float v[4 * kVClVec];
    cl_load_span(zrow, base, a.vec4t, a.V, v, flag);
    if (greedy) {
      unsigned long long best = ~0ull;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) {
        const int id = base + (e >> 2) * (kVClThreads * 4) + t * 4 + (e & 3);
        if (id < a.V) {
          const unsigned long long kk = zid_key(v[e], (unsigned int)id);
          best = kk < best ? kk : best;
        }
      }
      best = warp_min_u64(best);
      if (lane == 0) w.wkey[warp] = best;
      __syncthreads();
      if (warp == 0) {
        const unsigned long long kk = warp_min_u64(w.wkey[lane & (NW - 1)]);
        if (lane < R) cl_st_u64(cl_map(&w.gkey[par][q], (uint32_t)lane), kk);
      }
    } else {
      // the children's tokens leave this block's sums (the residual after every child is rejected)
      for (int x = t; x < kVClSpan / 32; x += kVClThreads) w.rejbits[x] = 0u;
      __syncthreads();
      if (nkid > 0) {
        mark_child_tokens(a, fo, w.kid, nkid, base, kVClSpan / 32, w.rejbits);
#pragma unroll
        for (int e = 0; e < 4 * kVClVec; ++e) {
          const int off = (e >> 2) * (kVClThreads * 4) + t * 4 + (e & 3);
          if ((w.rejbits[off >> 5] >> (off & 31)) & 1u) v[e] = -INFINITY;
        }
        pm_child_inputs(a, fo, w.kid, nkid, zrow, w.ktok, w.zk, w.uk);  // every CTA: the same inputs
      }
      float lm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) lm = fmaxf(lm, v[e]);
      lm = warp_max(lm);
      if (lane == 0) w.wmax[warp] = lm;
      __syncthreads();
      float Mq = w.wmax[0];
#pragma unroll
      for (int x = 1; x < NW; ++x) Mq = fmaxf(Mq, w.wmax[x]);
      float ls = 0.f;
      if (Mq > -INFINITY) {
#pragma unroll
        for (int e = 0; e < 4 * kVClVec; ++e) ls += exp_fast((v[e] - Mq) * invT);
      }
      ls = warp_sum(ls);
      if (lane == 0) w.wsum[warp] = ls;
      __syncthreads();
      if (t < R) {  // this block's pair into every block of the cluster
        float Sq = 0.f;
#pragma unroll
        for (int x = 0; x < NW; ++x) Sq += w.wsum[x];
        cl_st_f32x2(cl_map(&w.gms[par][q], (uint32_t)t), Mq, Sq);
      }
    }
    cl_arrive();  // release this block's stores
    cl_wait();    // every block's statistic is in every block
    int nxt = -1;
    if (greedy) {
      unsigned long long kk = w.gkey[par][0];
      for (int x = 1; x < R; ++x) kk = w.gkey[par][x] < kk ? w.gkey[par][x] : kk;
      am = (int)zid_id(kk);
      for (int k = 0; k < nkid && nxt < 0; ++k)
        if (w.tok[w.kid[k]] == am) nxt = w.kid[k];  // the first child (row order) with the argmax token
    } else {
      M = -INFINITY;
      for (int x = 0; x < R; ++x) M = fmaxf(M, w.gms[par][x].x);
      S = 0.f;
      for (int x = 0; x < R; ++x)  // the same order in every block: the same M and S
        S += w.gms[par][x].x > -INFINITY ? w.gms[par][x].y * expf((w.gms[par][x].x - M) * invT) : 0.f;
      if (warp == 0) {
        const int d = nkid > 0 ? pm_decide(nkid, w.kid, w.zk, w.uk, M, S, invT) : -1;
        if (lane == 0) w.s_acc = d;
      }
      __syncthreads();
      acc = w.s_acc;
      nxt = acc >= 0 ? acc : -1;
    }
    if (nxt < 0 || alen >= a.D) break;
    if (q == 0 && t == 0) {
      w.otok[alen] = w.tok[nxt];
      w.opath[alen + 1] = nxt;
    }
    ++alen;
    cur = nxt;
    __syncthreads();  // the step's shared arrays are rewritten by the next
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (q != 0) return;
  // ---- the leader: the bonus token at the stop row, then the outputs ----
  if (greedy) {
    if (t == 0) w.otok[alen] = am;
  } else {
    const int nrej = acc == -2 ? nkid : 0;  // every child of the stop row rejected: their tokens are out of the draw
    for (int k = t; k < nrej; k += kVClThreads) w.rej[k] = w.tok[w.kid[k]];
    __syncthreads();
    // the stop row's chunk statistics, into the workspace the draw reads them
    // from (through L2, as the parallel kernel's are)
    const int last = alen;  // the walk stopped in step alen (one step per accepted child, then the stop row)
    float *cst = a.part + (fo + cur) * (long long)a.nchunk * 2;
    for (int x = t; x < R; x += kVClThreads) {
      cst[2 * x] = w.gms[last & 1][x].x;
      cst[2 * x + 1] = w.gms[last & 1][x].y;
    }
    __syncthreads();
    const CdfRow cdf{kVClSpan, R, a.V, a.vec4t, a.T, invT};  // chunk maxima are raw logits
    const int bonus = bonus_from_chunks<kVClThreads, true>(cdf, zrow, cst, M, a.uniforms[fo], w.rej, nrej, w.redz,
                                                          w.redi, w.cdf_tsum, w.rejbits);
    if (t == 0) w.otok[alen] = bonus;
  }
  __syncthreads();
  const long long po = (long long)b * (a.D + 1);
  for (int j = t; j <= a.D; j += kVClThreads) {
    a.path[po + j] = j <= alen ? w.opath[j] : -1;
    a.tokens[po + j] = j <= alen ? w.otok[j] : -1;
  }
  if (t == 0) a.accept_len[b] = alen;
  if (badp && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
}

}  // namespace et

using namespace et;

extern "C" et_status et_verify_accept(const et_tree_cfg *cfg, et_accept_mode mode, const et_tree *tree,
                                      const float *target_logits, int64_t target_stride,
                                      const int32_t *target_row_of_node, const float *draft_logits,
                                      int64_t draft_stride, const int32_t *draft_row_of_node,
                                      const float *uniforms, int32_t *accept_len, int32_t *path, int32_t *tokens,
                                      int32_t *dev_status, void *ws, size_t ws_bytes, et_stream_t stream) {
  Geometry g;
  ET_RETURN_IF(!make_geometry(cfg, &g), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(mode != ET_ACCEPT_GREEDY && mode != ET_ACCEPT_STOCH_POINT && mode != ET_ACCEPT_STOCH_DRAFTQ,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!tree || !tree->flat_node || !tree->flat_tok || !tree->flat_parent, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!target_logits || target_stride < cfg->V || !et_aligned(target_logits, 4), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!accept_len || !path || !tokens, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(mode != ET_ACCEPT_GREEDY && !uniforms, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(mode == ET_ACCEPT_STOCH_DRAFTQ && (!draft_logits || draft_stride < cfg->V), ET_ERR_INVALID_ARG);
  size_t cnt_bytes, part_off, rowstat_off, dq_off;
  const size_t need = et_internal_tree_ws(cfg, &cnt_bytes, &part_off, &rowstat_off, &dq_off);
  ET_RETURN_IF(!ws || ws_bytes < need || !et_aligned(ws, 256), ET_ERR_WORKSPACE);
  const int N = cfg->n + 1;
  ET_RETURN_IF((long long)cfg->B * N > 65535, ET_ERR_UNSUPPORTED);
  {  // the logit tables: device, or page-locked host memory (rows read over the host link)
    const void *d = nullptr;
    ET_RETURN_IF(!et_internal_table_ptr(target_logits, &d), ET_ERR_INVALID_ARG);
    target_logits = static_cast<const float *>(d);
    if (draft_logits) {
      ET_RETURN_IF(!et_internal_table_ptr(draft_logits, &d), ET_ERR_INVALID_ARG);
      draft_logits = static_cast<const float *>(d);
    }
  }
  VerifyArgs a;
  a.mode = (int)mode;
  a.B = cfg->B; a.V = cfg->V; a.N = N; a.C = g.C; a.D = cfg->depth;
  a.nchunk = (cfg->V + kVChunk - 1) / kVChunk;
  a.T = cfg->temperature;
  a.tlog = target_logits; a.tstride = target_stride; a.tmap = target_row_of_node;
  a.dlog = draft_logits; a.dstride = draft_stride; a.dmap = draft_row_of_node;
  a.uniforms = uniforms;
  a.flat_node = tree->flat_node; a.flat_tok = tree->flat_tok; a.flat_parent = tree->flat_parent;
  a.accept_len = accept_len; a.path = path; a.tokens = tokens; a.dev_status = dev_status;
  unsigned char *base = static_cast<unsigned char *>(ws);
  const int rows = cfg->B * (cfg->m > N ? cfg->m : N);
  a.row_cnt = reinterpret_cast<unsigned int *>(base);
  a.seq_cnt = a.row_cnt + rows;
  a.part = reinterpret_cast<float *>(base + part_off);
  a.rowstat = reinterpret_cast<float *>(base + rowstat_off);
  a.dq = reinterpret_cast<float *>(base + dq_off);
  a.vec4t = et_aligned(target_logits, 16) && target_stride % 4 == 0;
  a.vec4d = draft_logits && et_aligned(draft_logits, 16) && draft_stride % 4 == 0;
  if (cfg->V <= kVClMaxV) {  // one cluster of ceil(V / 4096) CTAs per flat row
    const int R = (cfg->V + kVClSpan - 1) / kVClSpan;
    a.cdf_span = kVClSpan;
    a.cdf_nch = R;
    if (mode == ET_ACCEPT_STOCH_DRAFTQ)
      return et_launch(k_verify_cl<true>, dim3(R, cfg->B * N, 1), dim3(kVClThreads), 0, (cudaStream_t)stream, R, a);
    // The walk reads at most D + 1 of the N rows per sequence, one after the
    // other.  With a target table in host memory it was measured slower in a
    // serving loop (its dependent reads queue behind the next step's copies on
    // the host link), so small batches read every row in one round either way.
    if (cfg->B >= kSeqWalkMinB)
      return et_launch(k_verify_seq, dim3(R, cfg->B, 1), dim3(kVClThreads), 0, (cudaStream_t)stream, R, a);
    return et_launch(k_verify_cl<false>, dim3(R, cfg->B * N, 1), dim3(kVClThreads), 0, (cudaStream_t)stream, R, a);
  }
  a.cdf_span = kVChunk;
  a.cdf_nch = a.nchunk;
  return et_launch(k_verify, dim3(a.nchunk, cfg->B * N), dim3(kVThreads), 0, (cudaStream_t)stream, 0, a);
}
