// Lossless acceptance walk on sm_103a (EAGLE blog "大模型系列——论文解读：
// eagle/eagle2", sections 1.1 and 1.2: one target pass verifies the whole
// draft and the output distribution is unchanged, greedy or not).
//
// Phase 1 (all blocks): every flat row's target logits are streamed once with
// 128-bit loads, split over blocks; each block reduces its slice (argmax, or
// max and sum of exp at temperature T); the last block of a row merges them.
// Phase 2 (the last row-block of a sequence): walk the tree from the root,
// then draw the bonus token by an inverse CDF over the stopping row.
#include "et_common.cuh"
#include "et_cdf.cuh"

extern "C" __attribute__((visibility("hidden"))) size_t et_internal_tree_ws(const et_tree_cfg *cfg, size_t *cnt_bytes, size_t *part_off,
                                      size_t *rowstat_off);

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
  unsigned int *row_cnt, *seq_cnt;
  int vec4t;
  int cdf_span, cdf_nch;  // STOCH_POINT: chunk statistics (max, sum) of each row in part, span tokens each
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

// Inverse CDF over a row: smallest v with sum_{u<=v} w(u) > uni * sum_u w(u)
// (falls back to the last v with w(v) > 0).  `w(v)` must be non-negative and
// give the same value on every call.  Pass 1 walks the row in tiles of 4·NT
// tokens, four consecutive tokens per thread (coalesced), summing each tile
// per warp in fp32; one warp adds the tiles in fp64 and finds the tile where
// the cumulative sum crosses; pass 2 rescans that tile alone with an fp64
// block scan.
constexpr int kCdfTileMax = kMaxV / (256 * 4);  // tiles of the largest row at 256 threads

template <int NT, typename WF>
__device__ int block_inverse_cdf(int V, float uni, WF w, double *redd, int *redi, float *tpart, double *tsum) {
  static_assert(NT == 256, "tile bookkeeping sized for 256 threads");
  constexpr int NW = NT / 32, TILE = NT * 4;
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const int ntile = (V + TILE - 1) / TILE;
  int lastpos = -1;
  for (int tile = 0; tile < ntile; ++tile) {
    float sl = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = tile * TILE + 4 * t + j;
      if (v < V) {
        const float x = w(v);
        sl += x;
        if (x > 0.f) lastpos = v;
      }
    }
    sl = warp_sum(sl);
    if (lane == 0) tpart[tile * NW + wp] = sl;
  }
  if (t == 0) { redi[0] = 0x7fffffff; redi[1] = -1; redi[3] = -1; }
  __syncthreads();
  if (lastpos >= 0) atomicMax(&redi[1], lastpos);
  if (wp == 0) {
    double total = 0.0;
    for (int c0 = 0; c0 < ntile; c0 += 32) {
      const int tile = c0 + lane;
      double ts = 0.0;
      if (tile < ntile) {
#pragma unroll
        for (int x = 0; x < NW; ++x) ts += (double)tpart[tile * NW + x];
        tsum[tile] = ts;
      }
      total += warp_sum_d(ts);
    }
    const double thr = (double)uni * total;
    double run = 0.0;
    int J = -1;
    double before = 0.0;
    for (int c0 = 0; c0 < ntile && J < 0; c0 += 32) {
      const int tile = c0 + lane;
      const double ts = tile < ntile ? tsum[tile] : 0.0;
      double incl = ts;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned int hit = __ballot_sync(0xffffffffu, tile < ntile && run + incl > thr);
      if (hit) {
        const int l = __ffs(hit) - 1;
        J = c0 + l;
        before = run + __shfl_sync(0xffffffffu, incl, l) - __shfl_sync(0xffffffffu, ts, l);
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      redd[0] = before;
      redd[1] = thr;
      redi[2] = J;
    }
  }
  __syncthreads();
  const int J = redi[2];
  if (J >= 0) {  // pass 2: the crossing tile only
    float x[4];
    double mine = 0.0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = J * TILE + 4 * t + j;
      x[j] = v < V ? w(v) : 0.f;
      mine += (double)x[j];
    }
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) tsum[wp] = incl;  // the tile sums are no longer needed
    __syncthreads();
    double wbase = 0.0;
    for (int x2 = 0; x2 < wp; ++x2) wbase += tsum[x2];
    double run = redd[0] + wbase + incl - mine;
    const double thr = redd[1];
    int lastJ = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (x[j] > 0.f) lastJ = J * TILE + 4 * t + j;
      run += (double)x[j];
      if (x[j] > 0.f && run > thr) { atomicMin(&redi[0], J * TILE + 4 * t + j); break; }
    }
    if (lastJ >= 0) atomicMax(&redi[3], lastJ);
  }
  __syncthreads();
  // not crossed inside the tile (its two sums differ in the last bits): the
  // crossing is at its end, so take its last token of positive weight
  const int r = redi[0] != 0x7fffffff ? redi[0] : (redi[3] >= 0 ? redi[3] : redi[1]);
  __syncthreads();
  return r;
}

struct WalkSmem {
  float redz[32];
  int redi[32];
  double redd[32];
  float cdf_tpart[kCdfTileMax * 8];  // per tile, per warp sums of the inverse CDF
  double cdf_tsum[kCdfTileMax];
  int par[kMaxN], tokf[kMaxN], nodef[kMaxN];
  float rs0[kMaxN], rs1[kMaxN];  // per flat row: argmax id (bits) / max, -, / sum
  float zc[kMaxN];               // target logit of each row's token in its parent's row
  int opath[kMaxDepth + 2], otok[kMaxDepth + 2];
  int rej[kMaxTopk];
  float rejw[kMaxTopk];  // exp(z/T - M) of each rejected child at the stop row
  unsigned int rejbits[kMaxSpanWords];  // rejected children inside the chunk being scanned
  float uni[kMaxN];      // this sequence's uniforms
  float zsh[kMaxTopk];
  int s_next, s_nrej, s_cur, s_alen;
};

// Phase 2 of acceptance, run by the last row-block of sequence b: walk the
// kept tree from the root (children in ascending flat row), then draw or take
// the bonus token at the row where the walk stops.
template <int NT>
__device__ void verify_walk(const VerifyArgs &a, int b, WalkSmem &w) {
  const int t = threadIdx.x;
  int flag = 0;
  float *redz = w.redz;
  int *redi = w.redi;
  double *redd = w.redd;
  int *par = w.par, *tokf = w.tokf, *nodef = w.nodef, *rej = w.rej;
  float *zsh = w.zsh;
  int &s_next = w.s_next, &s_nrej = w.s_nrej, &s_cur = w.s_cur;
  const int N = a.N;
  const long long fo = (long long)b * N;
  for (int j = t; j < N; j += NT) {
    par[j] = a.flat_parent[fo + j];
    tokf[j] = a.flat_tok[fo + j];
    nodef[j] = a.flat_node[fo + j];
  }
  if (t == 0) s_cur = 0;
  if (a.mode != ET_ACCEPT_STOCH_DRAFTQ) {
    // ---- greedy / point-mass: everything the walk needs, fetched in parallel ----
    int badp = 0;
    for (int j = t; j < N; j += NT) {
      w.rs0[j] = ld_cg(a.rowstat + 2 * (fo + j));
      w.rs1[j] = ld_cg(a.rowstat + 2 * (fo + j) + 1);
      if (a.mode == ET_ACCEPT_STOCH_POINT) w.uni[j] = a.uniforms[fo + j];
      if (a.mode == ET_ACCEPT_STOCH_POINT && j > 0) {
        const int p = a.flat_parent[fo + j];
        const int x = a.flat_tok[fo + j];
        const float *zp = (p >= 0 && p < N) ? table_row(a.tlog, a.tstride, a.tmap, a.C, b, a.flat_node[fo + p], fo + p, badp)
                                            : nullptr;
        int f2 = 0;
        w.zc[j] = (zp && x >= 0 && x < a.V) ? sanitize_logit(zp[x], f2) : -INFINITY;
      }
    }
    __syncthreads();
    if (t < 32) {  // one warp walks: 32 candidate rows per ballot
      const int lane = t;
      int cur = 0, alen = 0, nrej = 0;
      if (lane == 0) w.opath[0] = 0;
      for (int iter = 0; iter <= a.D; ++iter) {
        int nxt = -1;
        nrej = 0;
        if (a.mode == ET_ACCEPT_GREEDY) {
          const int am = __float_as_int(w.rs0[cur]);
          for (int j0 = cur + 1; j0 < N; j0 += 32) {  // first row (ascending) that is a child with token am
            const int j = j0 + lane;
            const unsigned int hit = __ballot_sync(0xffffffffu, j < N && par[j] == cur && tokf[j] == am);
            if (hit) { nxt = j0 + __ffs(hit) - 1; break; }
          }
          if (nxt < 0 && lane == 0) w.otok[alen] = am;
        } else {
          const float M = w.rs0[cur], S = w.rs1[cur];
          float R = 0.f;
          for (int j0 = cur + 1; j0 < N && nxt < 0; j0 += 32) {
            const int j = j0 + lane;
            const bool child = j < N && par[j] == cur;
            // p(x) and the uniform of every child at once; R (the mass of the
            // siblings rejected before a child) as a prefix sum in row order
            const float wx = child ? expf(w.zc[j] / a.T - M) : 0.f;
            const float px = (child && S > 0.f) ? wx / S : 0.f;
            float incl = px;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            const float Rj = R + (incl - px);
            const bool acc = child && w.uni[j] < ((Rj < 1.f) ? px / (1.f - Rj) : INFINITY);
            const unsigned int kids = __ballot_sync(0xffffffffu, child);
            const unsigned int hit = __ballot_sync(0xffffffffu, acc);
            const unsigned int rejected = hit ? (kids & ((1u << (__ffs(hit) - 1)) - 1u)) : kids;
            if ((rejected >> lane) & 1u) {  // children before the accepted one, in row order
              const int slot = nrej + __popc(rejected & ((1u << lane) - 1u));
              if (slot < kMaxTopk) { rej[slot] = tokf[j]; w.rejw[slot] = wx; }
            }
            nrej += __popc(rejected);
            R += __shfl_sync(0xffffffffu, incl, 31);
            if (hit) nxt = j0 + __ffs(hit) - 1;
          }
          if (nrej > kMaxTopk) nrej = kMaxTopk;
        }
        if (nxt < 0 || alen >= a.D) break;
        if (lane == 0) {
          w.otok[alen] = tokf[nxt];
          w.opath[alen + 1] = nxt;
        }
        ++alen;
        cur = nxt;
      }
      if (lane == 0) {
        s_cur = cur;
        s_nrej = nrej;
        w.s_alen = alen;
      }
    }
    __syncthreads();
    const int alen = w.s_alen;
    if (a.mode == ET_ACCEPT_STOCH_POINT) {  // bonus token: inverse CDF of the residual at the stop row
      const int cur = s_cur, nrej = s_nrej;
      int badz = 0;
      const float *zr = table_row(a.tlog, a.tstride, a.tmap, a.C, b, nodef[cur], fo + cur, badz);
      const CdfRow cdf{a.cdf_span, a.cdf_nch, a.V, a.vec4t, a.T};
      const int bonus = bonus_from_chunks<NT>(cdf, zr, a.part + (fo + cur) * (long long)a.nchunk * 2, w.rs0[cur],
                                              w.uni[0], rej, w.rejw, nrej, redd, redi, w.cdf_tsum, w.rejbits);
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
    return;
  }
  __syncthreads();
  int alen = 0;
  int bonus = -1;
  int badw = 0;
  for (int iter = 0; iter <= a.D + 1; ++iter) {
    const int cur = s_cur;
    if (t == 0) a.path[(long long)b * (a.D + 1) + alen] = cur;
    if (t == 0) { s_next = -1; s_nrej = 0; }
    __syncthreads();
    const float *zr = table_row(a.tlog, a.tstride, a.tmap, a.C, b, nodef[cur], fo + cur, badw);
    if (a.mode == ET_ACCEPT_GREEDY) {
      const int am = __float_as_int(ld_cg(a.rowstat + 2 * (fo + cur)));
      if (t == 0) {  // children are the rows after cur whose parent is cur; first match wins
        int best = -1;
        for (int j = cur + 1; j < N; ++j)
          if (par[j] == cur && tokf[j] == am) { best = j; break; }
        s_next = best;
      }
      __syncthreads();
      bonus = am;
    } else if (a.mode == ET_ACCEPT_STOCH_POINT) {
      const float M = ld_cg(a.rowstat + 2 * (fo + cur)), S = ld_cg(a.rowstat + 2 * (fo + cur) + 1);
      if (t == 0 && zr) {
        float R = 0.f;
        int nrej = 0;
        for (int j = cur + 1; j < N; ++j) {
          if (par[j] != cur) continue;
          const int x = tokf[j];
          if (x < 0 || x >= a.V) { badw = 1; continue; }
          const float px = expf(sanitize_logit(zr[x], flag) / a.T - M) / S;
          const float ratio = (R < 1.f) ? px / (1.f - R) : INFINITY;
          const float u = a.uniforms[fo + j];
          if (u < ratio) { s_next = j; break; }
          R += px;
          if (nrej < kMaxTopk) rej[nrej++] = x;
        }
        s_nrej = nrej;
      }
      __syncthreads();
      if (s_next < 0) {
        const int nrej = s_nrej;
        bonus = block_inverse_cdf<NT>(a.V, a.uniforms[fo], [&](int vv) -> float {
          if (!zr) return 0.f;
          for (int q = 0; q < nrej; ++q)
            if (rej[q] == vv) return 0.f;
          int f2 = 0;
          const float y = sanitize_logit(zr[vv], f2) / a.T;
          return y > -INFINITY ? expf(y - M) : 0.f;
        }, redd, redi, w.cdf_tpart, w.cdf_tsum);
      }
    } else {  // ET_ACCEPT_STOCH_DRAFTQ
      const float M = ld_cg(a.rowstat + 2 * (fo + cur)), S = ld_cg(a.rowstat + 2 * (fo + cur) + 1);
      bool has_child = false;
      for (int j = cur + 1; j < N; ++j)
        if (par[j] == cur) { has_child = true; break; }
      float Mq = 0.f, Sq = 1.f;
      const float *qr = nullptr;
      if (has_child) {
        qr = table_row(a.dlog, a.dstride, a.dmap, a.C, b, nodef[cur], fo + cur, badw);
        float lm = -INFINITY;
        for (int vv = t; vv < a.V; vv += NT) {
          int f2 = 0;
          lm = fmaxf(lm, qr ? sanitize_logit(qr[vv], f2) / a.T : -INFINITY);
        }
        Mq = block_max<NT>(lm, redz);
        float ls = 0.f;
        for (int vv = t; vv < a.V; vv += NT) {
          int f2 = 0;
          const float y = qr ? sanitize_logit(qr[vv], f2) / a.T : -INFINITY;
          ls += y > -INFINITY ? expf(y - Mq) : 0.f;
        }
        Sq = block_sum<NT>(ls, redz);
      }
      // r_j(v): p(v) with j residual updates applied (zsh[i] = 1/Z_{i+1}, 0 = kept)
      int nz = 0;
      auto pval = [&](int vv) -> float {
        int f2 = 0;
        const float y = zr ? sanitize_logit(zr[vv], f2) / a.T : -INFINITY;
        return y > -INFINITY ? expf(y - M) / S : 0.f;
      };
      auto qval = [&](int vv) -> float {
        int f2 = 0;
        const float y = qr ? sanitize_logit(qr[vv], f2) / a.T : -INFINITY;
        return y > -INFINITY ? expf(y - Mq) / Sq : 0.f;
      };
      auto rval = [&](int vv, int upto) -> float {
        float r = pval(vv);
        if (upto > 0) {
          const float q = qval(vv);
          for (int s2 = 0; s2 < upto; ++s2)
            if (zsh[s2] > 0.f) r = fmaxf(r - q, 0.f) * zsh[s2];
        }
        return r;
      };
      for (int j = cur + 1; j < N; ++j) {
        if (par[j] != cur) continue;
        const int x = tokf[j];
        if (x < 0 || x >= a.V) { badw = 1; continue; }
        const float qx = qval(x);
        const float rx = rval(x, nz);
        const float ratio = qx <= 0.f ? 1.f : fminf(1.f, rx / qx);
        if (a.uniforms[fo + j] < ratio) { if (t == 0) s_next = j; break; }
        // residual update: Z = sum_v max(r(v) - q(v), 0)
        double loc = 0.0;
        for (int vv = t; vv < a.V; vv += NT) loc += (double)fmaxf(rval(vv, nz) - qval(vv), 0.f);
        const double Z = block_sum_d<NT>(loc, redd);
        __syncthreads();
        if (t == 0 && nz < kMaxTopk) zsh[nz] = Z > 0.0 ? (float)(1.0 / Z) : 0.f;
        __syncthreads();
        if (nz < kMaxTopk) ++nz;
      }
      __syncthreads();
      if (s_next < 0) {
        const int nzf = nz;
        bonus = block_inverse_cdf<NT>(a.V, a.uniforms[fo], [&](int vv) -> float { return rval(vv, nzf); }, redd, redi, w.cdf_tpart, w.cdf_tsum);
      }
    }
    __syncthreads();
    const int nxt = s_next;
    if (nxt < 0 || alen >= a.D) {
      if (nxt >= 0) bonus = -1;  // cannot happen: the tree is at most D deep
      if (t == 0) a.tokens[(long long)b * (a.D + 1) + alen] = bonus;
      break;
    }
    if (t == 0) {
      a.tokens[(long long)b * (a.D + 1) + alen] = tokf[nxt];
      s_cur = nxt;
    }
    ++alen;
    __syncthreads();
  }
  if (t == 0) {
    a.accept_len[b] = alen;
    for (int j = alen + 1; j <= a.D; ++j) {
      a.path[(long long)b * (a.D + 1) + j] = -1;
      a.tokens[(long long)b * (a.D + 1) + j] = -1;
    }
  }
  if (badw && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  (void)flag;
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
  } else {
    float lm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4 * kVVec; ++j) {
      v[j] = v[j] / a.T;
      lm = fmaxf(lm, v[j]);
    }
    const float Mc = block_max<kVThreads>(lm, redz);
    float ls = 0.f;
    if (Mc > -INFINITY) {
#pragma unroll
      for (int j = 0; j < 4 * kVVec; ++j) ls += v[j] > -INFINITY ? expf(v[j] - Mc) : 0.f;
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
      float cm = -INFINITY, cs = 0.f;
      if (t < a.nchunk) { cm = ld_cg(rp + 2 * t); cs = ld_cg(rp + 2 * t + 1); }
      const float M = block_max<kVThreads>(cm, redz);
      const float S = block_sum<kVThreads>((t < a.nchunk && cm > -INFINITY) ? cs * expf(cm - M) : 0.f, redz);
      if (t == 0) { a.rowstat[2 * row] = M; a.rowstat[2 * row + 1] = S; }
    }
  }
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.N, &sflag)) return;

  verify_walk<kVThreads>(a, b, w);
}

// ---------------------------------------------------------------------------
// phase 1 on a thread-block cluster per flat row (V <= 32768): CTA q reduces
// logits [4096 q, 4096 q + 4096) and stores its result straight into the
// leader's shared memory; after one cluster barrier the leader merges them
// and writes the row's statistic.
// ---------------------------------------------------------------------------
constexpr int kVClThreads = 256;
constexpr int kVClVec = 4;
constexpr int kVClSpan = kVClThreads * 4 * kVClVec;
constexpr int kVClMaxCtas = 8;
constexpr int kVClMaxV = kVClSpan * kVClMaxCtas;

__global__ void __launch_bounds__(kVClThreads) k_verify_cl(VerifyArgs a) {
  __shared__ WalkSmem w;
  __shared__ unsigned long long wkey[kVClThreads / 32], gkey[kVClMaxCtas];
  __shared__ float wmax[kVClThreads / 32], wsum[kVClThreads / 32];
  __shared__ float2 gms[kVClMaxCtas];
  __shared__ int sflag;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int R = gridDim.x;
  const int q = (int)cl_rank();
  const int row = blockIdx.y;
  const int b = row / a.N;
  cl_arrive_relaxed();  // phase 0: this block has started (waited on before any remote store)
  pdl_wait();           // the previous kernel in the stream has completed
  pdl_trigger();        // only now may the next kernel launch: at most one waits ahead
  int flag = 0, bad = 0;
  const int node = a.flat_node[row];
  const float *zrow = table_row(a.tlog, a.tstride, a.tmap, a.C, b, node, row, bad);
  const int base = q * kVClSpan;
  float v[4 * kVClVec];
#pragma unroll
  for (int u = 0; u < kVClVec; ++u) {
    const int e0 = base + u * kVClThreads * 4 + t * 4;
    if (zrow && a.vec4t && e0 + 3 < a.V) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < a.V) ? __ldg(zrow + e0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (e0 + j < a.V) v[4 * u + j] = sanitize_logit(v[4 * u + j], flag);
  }
  const bool greedy = a.mode == ET_ACCEPT_GREEDY;
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
  } else {
    float lm = -INFINITY;
    const float invT = 1.f / a.T;
#pragma unroll
    for (int e = 0; e < 4 * kVClVec; ++e) {
      v[e] = v[e] * invT;
      lm = fmaxf(lm, v[e]);
    }
    lm = warp_max(lm);
    if (lane == 0) wmax[warp] = lm;
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  __syncthreads();
  cl_wait();  // phase 0 done: every block of the cluster runs
  if (greedy) {
    if (warp == 0) {
      const unsigned long long kk = warp_min_u64(wkey[lane & (kVClThreads / 32 - 1)]);
      if (lane == 0) cl_st_u64(cl_map(&gkey[q], 0), kk);
    }
  } else {
    float Mq = wmax[0];
#pragma unroll
    for (int x = 1; x < kVClThreads / 32; ++x) Mq = fmaxf(Mq, wmax[x]);
    float ls = 0.f;
    if (Mq > -INFINITY) {
#pragma unroll
      for (int e = 0; e < 4 * kVClVec; ++e) ls += exp_fast(v[e] - Mq);
    }
    ls = warp_sum(ls);
    if (lane == 0) wsum[warp] = ls;
    __syncthreads();
    if (t == 0) {
      float Sq = 0.f;
#pragma unroll
      for (int x = 0; x < kVClThreads / 32; ++x) Sq += wsum[x];
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
      float M = -INFINITY;
      for (int x = 0; x < R; ++x) M = fmaxf(M, gms[x].x);
      float S = 0.f;
      for (int x = 0; x < R; ++x) S += gms[x].x > -INFINITY ? gms[x].y * expf(gms[x].x - M) : 0.f;
      a.rowstat[2 * row] = M;
      a.rowstat[2 * row + 1] = S;
      float *cst = a.part + (long long)row * a.nchunk * 2;  // chunk statistics for the bonus draw
      for (int x = 0; x < R; ++x) { cst[2 * x] = gms[x].x; cst[2 * x + 1] = gms[x].y; }
    }
  }
  if (!arrive_last(&a.seq_cnt[b], (unsigned)a.N, &sflag)) return;
  verify_walk<kVClThreads>(a, b, w);
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
  size_t cnt_bytes, part_off, rowstat_off;
  const size_t need = et_internal_tree_ws(cfg, &cnt_bytes, &part_off, &rowstat_off);
  ET_RETURN_IF(!ws || ws_bytes < need || !et_aligned(ws, 256), ET_ERR_WORKSPACE);
  const int N = cfg->n + 1;
  ET_RETURN_IF((long long)cfg->B * N > 65535, ET_ERR_UNSUPPORTED);
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
  a.vec4t = et_aligned(target_logits, 16) && target_stride % 4 == 0;
  if (cfg->V <= kVClMaxV) {  // one cluster of ceil(V / 4096) CTAs per flat row
    const int R = (cfg->V + kVClSpan - 1) / kVClSpan;
    a.cdf_span = kVClSpan;
    a.cdf_nch = R;
    return et_launch(k_verify_cl, dim3(R, cfg->B * N, 1), dim3(kVClThreads), 0, (cudaStream_t)stream, R, a);
  }
  a.cdf_span = kVChunk;
  a.cdf_nch = a.nchunk;
  return et_launch(k_verify, dim3(a.nchunk, cfg->B * N), dim3(kVThreads), 0, (cudaStream_t)stream, 0, a);
}
