// Shared helpers of the sm_103a EAGLE-2 tree kernels: limits, the node-id
// geometry, fixed-point path keys, 64-bit rank keys and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <float.h>
#include <math.h>

#include "eagle_tree.h"

namespace et {

constexpr int kMaxTopk = 32;
constexpr int kMaxM = 32;
constexpr int kMaxDepth = 16;
constexpr int kMaxN = 128;
constexpr int kMaxC = 4096;
constexpr int kMaxV = 262144;
constexpr int kIdBits = 12;                      // C <= 4096
constexpr long long kKeyMin = -((1LL << 52) - 1);  // saturation of path keys (-2^20 nats)

// Layer widths and id bases of the dynamic tree (EAGLE-2 article, expansion
// phase): layer 1 has k nodes; layer l+1 has min(m, width_l) * k.
struct Geometry {
  int C;
  int depth;
  int width[kMaxDepth + 1];    // width[0] = 1 (root)
  int base[kMaxDepth + 2];     // first id of layer l (l >= 1); base[D+1] = C
  int expanded[kMaxDepth];     // nodes expanded at layer l
};

inline bool make_geometry(const et_tree_cfg *cfg, Geometry *g) {
  if (!cfg) return false;
  if (cfg->B < 1 || cfg->depth < 1 || cfg->depth > kMaxDepth || cfg->topk < 1 ||
      cfg->topk > kMaxTopk || cfg->m < 1 || cfg->m > kMaxM || cfg->V < cfg->topk ||
      cfg->V > kMaxV || !(cfg->temperature > 0.f) || cfg->n < 1 || cfg->n + 1 > kMaxN)
    return false;
  g->depth = cfg->depth;
  g->width[0] = 1;
  g->width[1] = cfg->topk;
  long long C = cfg->topk;
  for (int l = 2; l <= cfg->depth; ++l) {
    int e = g->width[l - 1] < cfg->m ? g->width[l - 1] : cfg->m;
    g->width[l] = e * cfg->topk;
    C += g->width[l];
    if (C > kMaxC) return false;
  }
  g->C = (int)C;
  g->base[1] = 0;
  for (int l = 1; l <= cfg->depth; ++l) g->base[l + 1] = g->base[l] + g->width[l];
  g->base[0] = -1;
  g->expanded[0] = 1;
  for (int l = 1; l < cfg->depth; ++l) g->expanded[l] = g->width[l] < cfg->m ? g->width[l] : cfg->m;
  if (cfg->n > g->C) return false;
  return true;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
// NaN counts as -inf, +inf as FLT_MAX; reports either through *flag.
__device__ __forceinline__ float sanitize_logit(float z, int &flag) {
  if (z != z) { flag = 1; return -INFINITY; }
  if (z == INFINITY) { flag = 1; return FLT_MAX; }
  return z;
}

// (z desc, id asc): is (za, ia) ranked before (zb, ib)?
__device__ __forceinline__ bool ranks_before(float za, int ia, float zb, int ib) {
  return za > zb || (za == zb && ia < ib);
}

// Fixed-point image of an fp32 log-prob: rint(lp * 2^32), saturating.  The
// product lp * 2^32 is exact in fp32 (a power-of-two scale).
__device__ __forceinline__ long long fixed_key(float lp) {
  if (!(lp > -4.0e15f / 4294967296.0f)) return kKeyMin;  // -inf, NaN, or beyond the range
  long long k = __float2ll_rn(lp * 4294967296.0f);
  return k < kKeyMin ? kKeyMin : k;
}

__device__ __forceinline__ long long add_keys(long long a, long long b) {
  long long s = a + b;
  return s < kKeyMin ? kKeyMin : s;
}

// Unique 64-bit rank key: ascending order == (key desc, id asc).
__device__ __forceinline__ unsigned long long rank_key(long long key, int id) {
  if (key > 0) key = 0;
  if (key < kKeyMin) key = kKeyMin;
  return ((unsigned long long)(-key) << kIdBits) | (unsigned long long)id;
}

__device__ __forceinline__ void flag_status(int32_t *dev_status, int bits) {
  if (dev_status && bits) atomicOr(dev_status, bits);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// every lane gets the warp's smallest 64-bit value (two 32-bit reductions)
__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
  const unsigned int hi = (unsigned int)(v >> 32);
  const unsigned int mh = __reduce_min_sync(0xffffffffu, hi);
  const unsigned int ml = __reduce_min_sync(0xffffffffu, hi == mh ? (unsigned int)v : 0xffffffffu);
  return ((unsigned long long)mh << 32) | ml;
}
// warp-wide best (z desc, id asc); every lane gets the winner
__device__ __forceinline__ void warp_best(float &z, int &id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    int i2 = __shfl_xor_sync(0xffffffffu, id, o);
    if (ranks_before(z2, i2, z, id)) { z = z2; id = i2; }
  }
}

// Block reductions; `red` must hold >= 32 elements; all threads get the result.
template <int NT>
__device__ __forceinline__ float block_max(float v, float *red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < NT / 32 ? red[l] : -INFINITY;
  return warp_max(v);
}
template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < NT / 32 ? red[l] : 0.f;
  return warp_sum(v);
}
template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double *red) {
  v = warp_sum_d(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < NT / 32 ? red[l] : 0.0;
  return warp_sum_d(v);
}
template <int NT>
__device__ __forceinline__ unsigned long long block_min_u64(unsigned long long v, unsigned long long *red) {
  v = warp_min_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < NT / 32 ? red[l] : ~0ull;
  return warp_min_u64(v);
}
template <int NT>
__device__ __forceinline__ void block_best(float &z, int &id, float *redz, int *redi) {
  warp_best(z, id);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) { redz[w] = z; redi[w] = id; }
  __syncthreads();
  if (l < NT / 32) { z = redz[l]; id = redi[l]; } else { z = -INFINITY; id = 0x7fffffff; }
  warp_best(z, id);
}

// "Last block to arrive" handshake: every thread of the block has written its
// part; returns true in exactly one block per counter round and re-arms the
// counter for the next call.  No block ever waits on another.
__device__ __forceinline__ bool arrive_last(unsigned int *counter, unsigned int expected, int *smem_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned int prev = atomicAdd(counter, 1u);
    int last = (prev == expected - 1);
    if (last) *counter = 0u;  // all arrivals of this round are in
    *smem_flag = last;
  }
  __syncthreads();
  const bool last = *smem_flag != 0;
  if (last) __threadfence();
  return last;
}

template <typename T>
__device__ __forceinline__ T ld_cg(const T *p) { return __ldcg(p); }

// e^x for x <= 0 through the hardware base-2 exponential (used for sums of
// exponentials whose relative error budget is ~1e-6)
__device__ __forceinline__ float exp_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}

// ---- programmatic dependent launch ----
// Every kernel of this library but the persistent tree build is launched with
// programmatic stream serialization: it may start while the previous kernel
// in the stream is still running.  pdl_wait() blocks until that kernel has completed and its
// memory is visible, so it comes before the first global memory access;
// pdl_trigger() lets the next kernel start launching (it still waits for
// this one to complete before touching memory).  Triggering only after the
// wait keeps at most one kernel waiting ahead: triggering first lets a whole
// chain of launches pile up on the SMs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- thread-block clusters: distributed shared memory ----
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(const void *local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ float cl_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int cl_ld_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// split cluster barrier: arrive (release, or relaxed when it only has to
// show that every block of the cluster has started) ... wait (acquire)
__device__ __forceinline__ void cl_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_st_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void cl_st_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float a) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}
__device__ __forceinline__ void cl_st_f32x4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// ---- (value desc, id asc) as one ascending 64-bit key ----
// high word: the order-reversed image of z (larger z -> smaller word; -0 and
// +0 are one value), low word: the id.  Sanitised logits only (no NaN).
__device__ __forceinline__ unsigned long long zid_key(float z, unsigned int id) {
  if (z == 0.f) z = 0.f;  // -0 -> +0
  const unsigned int u = __float_as_uint(z);
  const unsigned int ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending with z
  return ((unsigned long long)(~ord) << 32) | id;
}
__device__ __forceinline__ float zid_value(unsigned long long key) {
  const unsigned int ord = ~(unsigned int)(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}
__device__ __forceinline__ unsigned int zid_id(unsigned long long key) { return (unsigned int)key; }

// (max, sum of exp(x - max)) pairs: merge two
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) { m = M; s = 0.f; return; }
  s = (m > -INFINITY ? s * exp_fast(m - M) : 0.f) + (m2 > -INFINITY ? s2 * exp_fast(m2 - M) : 0.f);
  m = M;
}

// Exact k smallest keys (k <= 32) of the NV keys each lane of a warp holds,
// ascending, into out[0..k) (shared memory).  Keys must be distinct.  The
// k-th smallest of the 32 lane minima bounds the answer from above (k lanes
// hold a key at or below it), so only keys at or below that bound compete;
// they are ranked by counting in `cand` (cap keys).  When more than cap keys
// compete (heavy ties), k rounds of warp argmin decide instead.
template <int NV>
__device__ __forceinline__ void warp_topk_keys(const unsigned long long (&key)[NV], int k, unsigned long long *cand,
                                               int cap, unsigned long long *out) {
  const int lane = threadIdx.x & 31;
  unsigned long long best = ~0ull;
#pragma unroll
  for (int e = 0; e < NV; ++e) best = key[e] < best ? key[e] : best;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) rank += __shfl_sync(0xffffffffu, best, j) < best ? 1 : 0;
  const unsigned int hit = __ballot_sync(0xffffffffu, rank == k - 1);
  const unsigned long long tau = __shfl_sync(0xffffffffu, best, __ffs(hit) - 1);
  int c = 0;
#pragma unroll
  for (int e = 0; e < NV; ++e) c += key[e] <= tau ? 1 : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int nc = __shfl_sync(0xffffffffu, incl, 31);
  if (nc <= cap) {
    int pos = incl - c;
#pragma unroll
    for (int e = 0; e < NV; ++e)
      if (key[e] <= tau) cand[pos++] = key[e];
    __syncwarp();
    for (int i = lane; i < nc; i += 32) {
      const unsigned long long mine = cand[i];
      int r = 0;
      for (int j0 = 0; j0 < nc; j0 += 8) {  // eight independent loads per round
#pragma unroll
        for (int j = j0; j < j0 + 8; ++j) r += (j < nc && cand[j] < mine) ? 1 : 0;
      }
      if (r < k) out[r] = mine;
    }
  } else {
    unsigned int used = 0u;
    for (int r = 0; r < k; ++r) {
      unsigned long long m = best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, m, o);
        m = w < m ? w : m;
      }
      if (lane == 0) out[r] = m;
      if (best == m) {
        best = ~0ull;
#pragma unroll
        for (int e = 0; e < NV; ++e) {
          if (key[e] == m) used |= 1u << e;
          if (!((used >> e) & 1u) && key[e] < best) best = key[e];
        }
      }
    }
  }
  __syncwarp();
}

// The n smallest of P distinct keys in shared memory, by rank: emit(r, key)
// runs once for each key of rank r < n.  Every thread of the block (NT
// threads) calls it.  Ranks are counted pairwise: G lanes share a key, each
// scanning every G-th key with eight independent loads per round, then a
// shuffle sum; G is the largest power of two (<= 32) with G * P <= NT.
template <int NT, typename Emit>
__device__ __forceinline__ void block_select(const unsigned long long *keys, int P, int n, Emit emit) {
  int G = 1;
  while (G < 32 && 2 * G * P <= NT) G *= 2;
  const int t = threadIdx.x;
  for (int base = 0; base < P * G; base += NT) {  // same trip count in every thread
    const int idx = base + t, i = idx / G, g = idx & (G - 1);
    const unsigned long long mine = i < P ? keys[i] : 0ull;
    int cnt = 0;
    if (i < P) {
      int j = g;
      for (; j + 7 * G < P; j += 8 * G) {
#pragma unroll
        for (int u = 0; u < 8; ++u) cnt += keys[j + u * G] < mine ? 1 : 0;
      }
      for (; j < P; j += G) cnt += keys[j] < mine ? 1 : 0;
    }
    for (int o = G >> 1; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (i < P && g == 0 && cnt < n) emit(cnt, mine);
  }
}

}  // namespace et

// host-side helpers shared by the entry points
#define ET_RETURN_IF(cond, code) \
  do {                           \
    if (cond) return (code);     \
  } while (0)

static inline et_status et_launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ET_OK : ET_ERR_CUDA;
}
static inline bool et_aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The bound, in SM clock cycles, of the device waits of the kernels launched
// from now on (et_set_wait_limit; defined in et_tree.cu).
__attribute__((visibility("hidden"))) long long et_wait_limit_cycles();

#include <mutex>
// Set a kernel attribute once per (kernel, attribute, device): the attribute
// lives in the current device's context, so every device that runs the
// kernel needs its own call.  Thread-safe.
static inline cudaError_t et_func_attr(const void *kernel, cudaFuncAttribute attr, int value) {
  static std::mutex mu;
  static const void *done_fn[64];
  static int done_attr[64];
  static int done_dev[64];
  static int ndone = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < ndone; ++i)
    if (done_fn[i] == kernel && done_attr[i] == (int)attr && done_dev[i] == dev) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, attr, value);
  if (e != cudaSuccess) return e;
  if (ndone < 64) {
    done_fn[ndone] = kernel;
    done_attr[ndone] = (int)attr;
    done_dev[ndone] = dev;
    ++ndone;
  }
  return cudaSuccess;
}
// Raise a kernel's dynamic shared-memory limit (once per kernel and device).
static inline cudaError_t et_smem_attr(const void *kernel, int bytes) {
  return et_func_attr(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Launch with programmatic stream serialization (pdl) or as a plain stream-
// ordered launch, and, when cluster_x > 0, in clusters of cluster_x blocks
// along x.
template <typename... KArgs, typename... Args>
static inline et_status et_launch_ex(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, int cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  if (cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return ET_ERR_CUDA;
  }
  return et_launch_status();
}
template <typename... KArgs, typename... Args>
static inline et_status et_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  int cluster_x, Args &&...args) {
  return et_launch_ex(true, kern, grid, block, smem, stream, cluster_x, static_cast<Args &&>(args)...);
}
