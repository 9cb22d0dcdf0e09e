// Static draft tree (EAGLE-1 / Medusa style; the EAGLE-2 article on
// sbmmt.com contrasts it with the dynamic tree): the tree's shape is fixed
// in advance as flat rows -- row 0 the root, row i > 0 with a parent row
// parent[i] < i and a rank rank[i] -- and row i's token is the rank[i]-th best
// token (largest draft logit first, lower id on ties) of the draft logits at
// its parent.  The output is the same flattened tree the dynamic path
// produces, so the mask, attention and acceptance calls run unchanged.
//
// One thread-block cluster of ceil(V / 4096) blocks per (sequence, flat row)
// that has children: every warp finds the exact top-k of its 512 logits,
// each block selects its top-k from its warps' lists and stores it into the
// leader's shared memory, and after one cluster barrier the leader selects
// the row's top-k and hands each child its ranked token.  Rows without
// children only write their own flat entries.
#include "et_common.cuh"
#include "et_cdf.cuh"

namespace et {
namespace {

constexpr int kStThreads = 256;
constexpr int kStWarps = kStThreads / 32;
constexpr int kStVec = 4;
constexpr int kStSpan = kStThreads * 4 * kStVec;  // 4096 logits per block
constexpr int kStMaxCtas = 8;
constexpr int kStWarpCand = 64;

struct StaticArgs {
  int B, V, N, k, vec4;
  const int32_t *parent, *rank;  // [N]
  const float *logits;
  long long row_stride;
  const int32_t *row_of_flat;    // [B, N]
  const int32_t *root_tok;       // [B] or null
  int32_t *flat_tok, *flat_parent, *flat_depth, *flat_node;
  int32_t *dev_status;
};

struct StaticSmem {
  unsigned long long cand[kStWarps][kStWarpCand];
  unsigned long long wl[kStWarps * kMaxTopk];
  unsigned long long gl[kStMaxCtas * kMaxTopk];
  unsigned long long top[kMaxTopk];
  int par[kMaxN], rk[kMaxN];
  int has_child;
};

__global__ void __launch_bounds__(kStThreads) k_static_cl(StaticArgs a) {
  __shared__ StaticSmem sh;
  const int t = threadIdx.x, warp = t >> 5;
  const int q = (int)cl_rank();
  const int i = blockIdx.y % a.N, b = blockIdx.y / a.N;
  const int k = a.k;
  cl_arrive_relaxed();  // phase 0: this block has started (waited on before any remote store)
  pdl_wait();           // the previous kernel in the stream has completed
  pdl_trigger();        // only now may the next kernel launch: at most one waits ahead
  if (t == 0) sh.has_child = 0;
  for (int j = t; j < a.N; j += kStThreads) {
    sh.par[j] = a.parent[j];
    sh.rk[j] = a.rank[j];
  }
  __syncthreads();
  for (int j = i + 1 + t; j < a.N; j += kStThreads)
    if (sh.par[j] == i) sh.has_child = 1;
  __syncthreads();
  const long long fo = (long long)b * a.N;
  if (q == 0 && t == 0) {  // this row's own flat entries
    int d = 0, j = i, bad = 0;
    while (j > 0 && d <= kMaxN) {
      const int p = sh.par[j];
      if (p < 0 || p >= j) { bad = 1; break; }
      j = p;
      ++d;
    }
    if (i == 0 && sh.par[0] != -1) bad = 1;
    a.flat_parent[fo + i] = i == 0 ? -1 : sh.par[i];
    a.flat_node[fo + i] = i - 1;
    a.flat_depth[fo + i] = d;
    if (i == 0) a.flat_tok[fo] = a.root_tok ? a.root_tok[b] : -1;
    if (bad) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  }
  if (!sh.has_child) return;  // the same for every block of the cluster

  int flag = 0, bad = 0;
  const int r = a.row_of_flat[fo + i];
  const float *zrow = r >= 0 ? a.logits + (long long)r * a.row_stride : nullptr;
  if (r < 0) bad = 1;
  const int base = q * kStSpan;
  float v[4 * kStVec];
#pragma unroll
  for (int u = 0; u < kStVec; ++u) {
    const int e0 = base + u * kStThreads * 4 + t * 4;
    if (zrow && a.vec4 && e0 + 3 < a.V) {
      const float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < a.V) ? __ldcs(zrow + e0 + j) : -INFINITY;
    }
  }
  unsigned long long key[4 * kStVec];
#pragma unroll
  for (int u = 0; u < kStVec; ++u) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * u + j, id = base + u * kStThreads * 4 + t * 4 + j;  // ids >= V are padding
      if (id < a.V) v[e] = sanitize_logit(v[e], flag);
      key[e] = zid_key(v[e], (unsigned int)id);
    }
  }
  warp_topk_keys<4 * kStVec>(key, k, sh.cand[warp], kStWarpCand, sh.wl + warp * k);
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
  if (bad && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  __syncthreads();
  cl_wait();  // phase 0 done: every block of the cluster runs
  const uint32_t gl_remote = cl_map(&sh.gl[q * k], 0);
  block_select<kStThreads>(sh.wl, kStWarps * k, k,
                           [&](int rr, unsigned long long kr) { cl_st_u64(gl_remote + 8u * (uint32_t)rr, kr); });
  cl_arrive();  // phase 1: release this block's stores
  if (q != 0) return;
  cl_wait();
  block_select<kStThreads>(sh.gl, (int)gridDim.x * k, k, [&](int rr, unsigned long long kr) { sh.top[rr] = kr; });
  __syncthreads();
  for (int c = i + 1 + t; c < a.N; c += kStThreads) {
    if (sh.par[c] != i) continue;
    const int rc = sh.rk[c];
    int tok = -1;
    if (rc >= 0 && rc < k && zrow) {
      const int id = (int)zid_id(sh.top[rc]);
      tok = id < a.V ? id : -1;
    } else {
      flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    }
    a.flat_tok[fo + c] = tok;
  }
}

// ---------------------------------------------------------------------------
// sampled children (the proposal the draft-q acceptance rule needs): row i's
// token is an independent draw from q = softmax(draft / T) at its parent, by
// inverse CDF with uniforms[b, i].  Pass 1: (max, sum of exp) of every
// 4096-token chunk of every row that has children; pass 2: one block per
// child row finds the chunk where u * total falls and rescans it.
// ---------------------------------------------------------------------------
struct SampledArgs {
  int B, V, N, R, vec4;
  float T;
  const int32_t *parent;
  const float *logits;
  long long row_stride;
  const int32_t *row_of_flat;
  const int32_t *root_tok;
  const float *uniforms;    // [B, N]
  float *cst;               // [B, N, R] (max, sum) pairs
  int32_t *flat_tok, *flat_parent, *flat_depth, *flat_node;
  int32_t *dev_status;
};

__global__ void __launch_bounds__(kStThreads) k_static_stats(SampledArgs a) {
  __shared__ int par[kMaxN];
  __shared__ int has_child;
  __shared__ float red[32];
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  const int t = threadIdx.x, q = blockIdx.x;
  const int i = blockIdx.y % a.N, b = blockIdx.y / a.N;
  if (t == 0) has_child = 0;
  for (int j = t; j < a.N; j += kStThreads) par[j] = a.parent[j];
  __syncthreads();
  for (int j = i + 1 + t; j < a.N; j += kStThreads)
    if (par[j] == i) has_child = 1;
  __syncthreads();
  const long long fo = (long long)b * a.N;
  if (q == 0 && t == 0) {  // this row's own flat entries
    int d = 0, j = i, bad = 0;
    while (j > 0 && d <= kMaxN) {
      const int p = par[j];
      if (p < 0 || p >= j) { bad = 1; break; }
      j = p;
      ++d;
    }
    if (i == 0 && par[0] != -1) bad = 1;
    a.flat_parent[fo + i] = i == 0 ? -1 : par[i];
    a.flat_node[fo + i] = i - 1;
    a.flat_depth[fo + i] = d;
    if (i == 0) a.flat_tok[fo] = a.root_tok ? a.root_tok[b] : -1;
    if (bad) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  }
  if (!has_child) return;
  const int r = a.row_of_flat[fo + i];
  const float *zrow = r >= 0 ? a.logits + (long long)r * a.row_stride : nullptr;
  if (r < 0 && q == 0 && t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  const int base = q * kStSpan;
  const float invT = 1.f / a.T;
  float v[4 * kStVec];
  int flag = 0;
  float lm = -INFINITY;
#pragma unroll
  for (int u = 0; u < kStVec; ++u) {
    const int e0 = base + u * kStThreads * 4 + t * 4;
    if (zrow && a.vec4 && e0 + 3 < a.V) {
      const float4 f = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
      v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[4 * u + j] = (zrow && e0 + j < a.V) ? __ldcs(zrow + e0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (e0 + j < a.V) v[4 * u + j] = sanitize_logit(v[4 * u + j], flag);
      v[4 * u + j] *= invT;
      lm = fmaxf(lm, v[4 * u + j]);
    }
  }
  const float Mq = block_max<kStThreads>(lm, red);
  float ls = 0.f;
  if (Mq > -INFINITY) {
#pragma unroll
    for (int e = 0; e < 4 * kStVec; ++e) ls += exp_fast(v[e] - Mq);  // as the acceptance walk's chunk sums
  }
  const float Sq = block_sum<kStThreads>(ls, red);
  if (t == 0) {
    float *c = a.cst + ((fo + i) * a.R + q) * 2;
    c[0] = Mq;
    c[1] = Sq;
  }
  if (flag) flag_status(a.dev_status, ET_DEV_NONFINITE);
}

__global__ void __launch_bounds__(kStThreads) k_static_draw(SampledArgs a) {
  __shared__ float redf[32], tsum[32];
  __shared__ int redi[32];
  __shared__ unsigned int rejbits[kMaxSpanWords];
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  const int i = blockIdx.x % a.N, b = blockIdx.x / a.N;
  if (i == 0) return;
  const long long fo = (long long)b * a.N;
  const int p = a.parent[i];
  if (p < 0 || p >= i) {
    if (threadIdx.x == 0) { a.flat_tok[fo + i] = -1; flag_status(a.dev_status, ET_DEV_BAD_INDEX); }
    return;
  }
  const int r = a.row_of_flat[fo + p];
  const float *zr = r >= 0 ? a.logits + (long long)r * a.row_stride : nullptr;
  const float *cst = a.cst + (fo + p) * a.R * 2;
  float M = -INFINITY;
  for (int x = 0; x < a.R; ++x) M = fmaxf(M, ld_cg(cst + 2 * x));
  const CdfRow cdf{kStSpan, a.R, a.V, a.vec4, a.T, 1.f};  // statistics of z / T
  const int tok = bonus_from_chunks<kStThreads, false>(cdf, zr, cst, M, a.uniforms[fo + i], nullptr, 0, redf, redi,
                                                       tsum, rejbits);
  if (threadIdx.x == 0) a.flat_tok[fo + i] = tok;
}

}  // namespace
}  // namespace et

using namespace et;

extern "C" size_t et_static_tree_workspace_size(const et_static_cfg *cfg) {
  if (!cfg || cfg->B < 1 || cfg->N < 1 || cfg->V < 1) return 0;
  const long long R = (cfg->V + kStSpan - 1) / kStSpan;
  return (((size_t)cfg->B * cfg->N * R * 2 * sizeof(float)) + 255) & ~(size_t)255;
}

extern "C" et_status et_static_tree_sampled(const et_static_cfg *cfg, const int32_t *parent, const float *logits,
                                            int64_t row_stride, const int32_t *row_of_flat, const float *uniforms,
                                            et_tree *tree, int32_t *dev_status, void *ws, size_t ws_bytes,
                                            et_stream_t stream) {
  ET_RETURN_IF(!cfg, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(cfg->B < 1 || cfg->N < 1 || cfg->N > kMaxN || cfg->V < 1 || !(cfg->temperature > 0.f) ||
                   (long long)cfg->B * cfg->N > 65535,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(cfg->V > kStSpan * kStMaxCtas, ET_ERR_UNSUPPORTED);
  ET_RETURN_IF(!parent || !logits || row_stride < cfg->V || !row_of_flat || !uniforms || !tree || !tree->flat_tok ||
                   !tree->flat_parent || !tree->flat_depth || !tree->flat_node,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  const size_t need = et_static_tree_workspace_size(cfg);
  ET_RETURN_IF(!ws || ws_bytes < need || !et_aligned(ws, 256), ET_ERR_WORKSPACE);
  SampledArgs a;
  a.B = cfg->B; a.V = cfg->V; a.N = cfg->N; a.R = (cfg->V + kStSpan - 1) / kStSpan;
  a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
  a.T = cfg->temperature;
  a.parent = parent; a.logits = logits; a.row_stride = row_stride; a.row_of_flat = row_of_flat;
  a.root_tok = tree->root_tok; a.uniforms = uniforms;
  a.cst = static_cast<float *>(ws);
  a.flat_tok = tree->flat_tok; a.flat_parent = tree->flat_parent; a.flat_depth = tree->flat_depth;
  a.flat_node = tree->flat_node;
  a.dev_status = dev_status;
  const et_status st = et_launch(k_static_stats, dim3(a.R, cfg->B * cfg->N), dim3(kStThreads), 0,
                                 (cudaStream_t)stream, 0, a);
  if (st != ET_OK) return st;
  return et_launch(k_static_draw, dim3(cfg->B * cfg->N), dim3(kStThreads), 0, (cudaStream_t)stream, 0, a);
}

extern "C" et_status et_static_tree(const et_static_cfg *cfg, const int32_t *parent, const int32_t *rank,
                                    const float *logits, int64_t row_stride, const int32_t *row_of_flat,
                                    et_tree *tree, int32_t *dev_status, et_stream_t stream) {
  ET_RETURN_IF(!cfg, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(cfg->B < 1 || cfg->N < 1 || cfg->N > kMaxN || cfg->topk < 1 || cfg->topk > kMaxTopk ||
                   cfg->V < cfg->topk || (long long)cfg->B * cfg->N > 65535,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(cfg->V > kStSpan * kStMaxCtas, ET_ERR_UNSUPPORTED);
  ET_RETURN_IF(!parent || !rank || !logits || row_stride < cfg->V || !row_of_flat || !tree || !tree->flat_tok ||
                   !tree->flat_parent || !tree->flat_depth || !tree->flat_node,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  StaticArgs a;
  a.B = cfg->B; a.V = cfg->V; a.N = cfg->N; a.k = cfg->topk;
  a.vec4 = et_aligned(logits, 16) && (row_stride % 4 == 0);
  a.parent = parent; a.rank = rank; a.logits = logits; a.row_stride = row_stride; a.row_of_flat = row_of_flat;
  a.root_tok = tree->root_tok;
  a.flat_tok = tree->flat_tok; a.flat_parent = tree->flat_parent; a.flat_depth = tree->flat_depth;
  a.flat_node = tree->flat_node;
  a.dev_status = dev_status;
  const int R = (cfg->V + kStSpan - 1) / kStSpan;
  return et_launch(k_static_cl, dim3(R, cfg->B * cfg->N, 1), dim3(kStThreads), 0, (cudaStream_t)stream, R, a);
}
