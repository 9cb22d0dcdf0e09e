// Inverse CDF of a row from its chunk statistics: the row's tokens are split
// in chunks of `span` tokens whose weights (Mc, Sc) are already known, so one
// warp finds the chunk where the cumulative weight crosses uni * total and the
// block rescans that chunk alone.  Shared by the bonus draws of the acceptance
// walk and the sampled static tree.
#pragma once

#include "et_common.cuh"

namespace et {
namespace {

struct CdfRow {
  int span, nch, V, vec4;  // chunk tokens, chunks, vocabulary, 16-byte aligned row
  float T;                 // temperature
  float cscale;            // chunk c weighs Sc * exp((Mc - M) * cscale): 1 when the maxima are of z / T,
                           // 1 / T when they are of the raw logits z
};

constexpr int kMaxSpan = 4096;                  // chunk tokens (the clustered phase 1)
constexpr int kMaxSpanWords = kMaxSpan / 32;
constexpr int kMaxPer = kMaxSpan / 256;         // tokens per thread in the chunk pass
// Chunk c holds tokens [c·span, (c+1)·span) with statistics (Mc, Sc) that
// already leave out the rejected tokens: its weight is Sc·exp((Mc − M)·cscale),
// a sum of positive terms (nothing is subtracted).  The rescan weighs token v
// as wf(zt, zd), zt and zd its sanitised target and draft logits (zd = −inf
// without a draft row), and each of the nrej rejected tokens rej[] as 0; wf
// must give the weights the chunk statistics sum.  Sums are fp32 (the weights
// themselves are fp32 values with ~1e-7 relative error); the threshold inside
// the crossing chunk is taken relative to the chunk's start.
template <int NT, bool kDraft, typename WF>
__device__ int chunk_inverse_cdf(const CdfRow &a, const float *zr, const float *dr, int vec4d, const float *cstat,
                                 float M, float uni, const int *rej, int nrej, float *redf, int *redi, float *tsum,
                                 unsigned int *rejbits, WF wf) {
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const int span = a.span, nch = a.nch;
  if (t == 0) { redi[0] = 0x7fffffff; redi[1] = -1; }
  if (wp == 0) {
    float total = 0.f;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int c = c0 + lane;
      float wc = 0.f;
      if (c < nch) {
        const float mc = ld_cg(cstat + 2 * c), sc = ld_cg(cstat + 2 * c + 1);
        wc = mc > -INFINITY ? sc * expf((mc - M) * a.cscale) : 0.f;
        tsum[c] = wc;
      }
      total += warp_sum(wc);
    }
    const float thr = uni * total;
    float run = 0.f, rel = 0.f;
    int J = -1, lastc = -1;
    for (int c0 = 0; c0 < nch; c0 += 32) {
      const int c = c0 + lane;
      const float wc = c < nch ? tsum[c] : 0.f;
      float incl = wc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned int pos = __ballot_sync(0xffffffffu, c < nch && wc > 0.f);
      if (pos) lastc = c0 + 31 - __clz(pos);
      const unsigned int hit = __ballot_sync(0xffffffffu, c < nch && wc > 0.f && run + incl > thr);
      if (hit && J < 0) {
        const int l = __ffs(hit) - 1;
        J = c0 + l;
        rel = thr - (run + __shfl_sync(0xffffffffu, incl, l) - __shfl_sync(0xffffffffu, wc, l));
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (J < 0) {  // thr at or beyond the total (rounding): the last chunk with weight
      J = lastc;
      rel = -1.f;
    }
    if (lane == 0) {
      redf[0] = rel;  // the threshold relative to chunk J's start; < 0: take its last token
      redi[2] = J;
    }
  }
  // the rejected children inside a chunk, as a bitmap (span <= 4096 bits)
  for (int x = t; x < kMaxSpanWords; x += NT) rejbits[x] = 0u;
  __syncthreads();
  const int J = redi[2];
  if (J < 0 || !zr) {
    __syncthreads();
    return -1;
  }
  for (int q = t; q < nrej; q += NT) {
    const int off = rej[q] - J * span;
    if (off >= 0 && off < span) atomicOr(&rejbits[off >> 5], 1u << (off & 31));
  }
  __syncthreads();
  // pass over chunk J: per thread a contiguous run of span / NT (<= 16) tokens, kept in registers
  const int per = span / NT;
  const int v0 = J * span + t * per;
  float x[kMaxPer];
  float mine = 0.f;
  int lastv = -1;
#pragma unroll
  for (int j = 0; j < kMaxPer; j += 4) {
    float z4[4];
    if (j < per && a.vec4 && v0 + j + 3 < a.V) {
      const float4 f = *reinterpret_cast<const float4 *>(zr + v0 + j);
      z4[0] = f.x; z4[1] = f.y; z4[2] = f.z; z4[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) z4[e] = (j + e < per && v0 + j + e < a.V) ? zr[v0 + j + e] : -INFINITY;
    }
    float d4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (kDraft && dr) {
      if (j < per && vec4d && v0 + j + 3 < a.V) {
        const float4 f = *reinterpret_cast<const float4 *>(dr + v0 + j);
        d4[0] = f.x; d4[1] = f.y; d4[2] = f.z; d4[3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) d4[e] = (j + e < per && v0 + j + e < a.V) ? dr[v0 + j + e] : -INFINITY;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int jj = j + e, off = t * per + jj;
      int f2 = 0;
      const float zt = sanitize_logit(z4[e], f2);
      const float zd = kDraft ? sanitize_logit(d4[e], f2) : -INFINITY;
      const bool rejected = jj < per && ((rejbits[off >> 5] >> (off & 31)) & 1u);
      x[jj] = (jj < per && !rejected) ? wf(zt, zd) : 0.f;
      mine += x[jj];
      if (x[jj] > 0.f) lastv = v0 + jj;
    }
  }
  float incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) tsum[wp] = incl;  // the chunk weights are no longer needed
  if (lastv >= 0) atomicMax(&redi[1], lastv);
  __syncthreads();
  const float relJ = redf[0];
  if (relJ >= 0.f) {
    float wbase = 0.f;
    for (int x2 = 0; x2 < wp; ++x2) wbase += tsum[x2];
    // the threshold relative to this thread's run, then a walk over its tokens
    const float rel = relJ - (wbase + (incl - mine));
    if (rel < mine) {
      float run = 0.f;
#pragma unroll
      for (int jj = 0; jj < kMaxPer; ++jj) {
        if (jj >= per) break;
        run += x[jj];
        if (x[jj] > 0.f && run > rel) { atomicMin(&redi[0], v0 + jj); break; }
      }
    }
  }
  __syncthreads();
  // not crossed inside the chunk (its two sums differ in the last bits): the
  // crossing is at its end, so take its last token of positive weight
  const int r = redi[0] != 0x7fffffff ? redi[0] : redi[1];
  __syncthreads();
  return r;
}

// The inverse CDF of the softmax row p at temperature T (rejected tokens
// removed) from its chunk statistics.  kRaw: the statistics are (max of z,
// sum of exp((z − max)/T)) and M is a raw logit (a.cscale = 1/T); otherwise
// (max of z/T, sum of exp(z/T − max)) and M is a scaled logit (a.cscale = 1).
template <int NT, bool kRaw>
__device__ int bonus_from_chunks(const CdfRow &a, const float *zr, const float *cstat, float M, float uni,
                                 const int *rej, int nrej, float *redf, int *redi, float *tsum,
                                 unsigned int *rejbits) {
  const float invT = 1.f / a.T;
  return chunk_inverse_cdf<NT, false>(a, zr, nullptr, 0, cstat, M, uni, rej, nrej, redf, redi, tsum, rejbits,
                                      [&](float zt, float) -> float {  // as the chunk sums weigh it
                                        if (!(zt > -INFINITY)) return 0.f;
                                        return kRaw ? exp_fast((zt - M) * invT) : exp_fast(zt * invT - M);
                                      });
}

}  // namespace
}  // namespace et
