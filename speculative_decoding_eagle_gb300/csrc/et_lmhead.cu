// Draft LM head on the 5th-generation tensor cores (tcgen05) of sm_103a: the
// draft model's features of the nodes being expanded are turned into logits
// over the vocabulary by the target's LM head (EAGLE blog section 1.2: the
// draft reuses the target's embedding and LM head; one extra decoder layer
// produces the features), logits[m, v] = sum_h X[m, h] W[v, h].  The logits
// rows feed et_tree_expand (log-softmax, top-k, path values).
//
// With a few feature rows and V x H weights (32000 x 4096 bf16 = 262 MB) the
// product is bound by streaming W once, so the operands are swapped: a block
// owns 128 vocabulary rows of W as the MMA's M side and all feature rows
// (padded to N = 16, 32 or 64) as its N side, D = W_tile X^T in TMEM.
//   warp 0   TMA producer: 64-element k slices of W (128 x 128 B) and X
//            (N x 128 B), 128-byte swizzle, an S-stage ring (mbarrier
//            expect-tx / commit);
//   warp 1   owns the TMEM columns and issues tcgen05.mma (K = 16 per MMA,
//            four per k slice);
//   warps 0-3 read their TMEM lane quarter (32 vocabulary rows x N fp32)
//            after the last commit and write coalesced logits rows.
// Every wait is bounded; on expiry the block sets ET_DEV_TIMEOUT, drains its
// copies, frees its TMEM and returns.
#include "et_common.cuh"
#include "et_tc.cuh"

namespace et {
namespace {

constexpr int kLmThreads = 128;
constexpr int kLmRows = 128;                       // vocabulary rows per block (MMA M)
constexpr int kLmK = 64;                           // k elements per slice (128 bytes of bf16)
constexpr uint32_t kLmABytes = kLmRows * 128;      // one W slice
constexpr int kLmMaxN = 64;
// stages by padded N: 6 x (16 + 2) KB, 5 x (16 + 4) KB, 4 x (16 + 8) KB; two blocks fit per SM
constexpr int kLmSmemMax = 6 * (kLmABytes + 16 * 128) + 8 * 13 + 32 + 1024;

struct LmArgs {
  int M, Mp, H, V, stages;
  long long ldo;
  float *out;
  int32_t *dev_status;
  long long wait_cycles;  // bound of every mbarrier wait (et_set_wait_limit)
};

__global__ void __launch_bounds__(kLmThreads)
    k_lmhead_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, const LmArgs a) {
  pdl_wait();  // the previous kernel in the stream has completed (the features may come from it)
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = saddr(sm);
  const int S = a.stages;
  const uint32_t bBytes = (uint32_t)a.Mp * 128u;
  const uint32_t offB = (uint32_t)S * kLmABytes;
  const uint32_t offBar = offB + (uint32_t)S * bBytes;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + offBar + 8 * (2 * S + 1));
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + offBar + 8 * (2 * S + 1) + 16);
  auto full = [&](int s) -> uint32_t { return sb + offBar + 8u * (uint32_t)s; };
  auto empty = [&](int s) -> uint32_t { return sb + offBar + 8u * (uint32_t)(S + s); };
  const uint32_t done = sb + offBar + 8u * (uint32_t)(2 * S);
  const uint32_t drain = sb + offBar + 8u * (uint32_t)(2 * S + 1) + 24u;  // every issued MMA has finished
  const uint32_t tcols = a.Mp <= 32 ? 32u : 64u;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int v0 = blockIdx.x * kLmRows;
  const int nk = a.H / kLmK;
  if (t == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(tcols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();  // only now: a waiting dependent block must not hold the TMEM this block needs

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % S;
      if (kb >= S && !mbar_wait(empty(s), (uint32_t)((kb / S) - 1) & 1u, abort_flag, a.wait_cycles)) break;
      mbar_expect_tx(full(s), kLmABytes + bBytes);
      tma_2d(sb + (uint32_t)s * kLmABytes, &tm_w, kb * kLmK, v0, full(s));
      tma_2d(sb + offB + (uint32_t)s * bBytes, &tm_x, kb * kLmK, 0, full(s));
      issued = kb + 1;
    }
    const int first = issued > S ? issued - S : 0;  // copies not yet consumed may still be in flight
    for (int kb = first; kb < issued; ++kb) mbar_drain(full(kb % S), (uint32_t)(kb / S) & 1u);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16(kLmRows, a.Mp, false);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % S;
      if (!mbar_wait(full(s), (uint32_t)(kb / S) & 1u, abort_flag, a.wait_cycles)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kLmK / 16; ++kk) {
        const uint64_t ad = sw128_desc(sb + (uint32_t)s * kLmABytes + kk * 32, 16, 1024);
        const uint64_t bd = sw128_desc(sb + offB + (uint32_t)s * bBytes + kk * 32, 16, 1024);
        tc_mma(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(empty(s));  // the slice is consumed once its MMAs are done
    }
    if (ok) tc_commit(done);
    // TMEM is freed only after every MMA this thread issued has finished
    // (after an expired wait the epilogue does not wait for them)
    tc_commit(drain);
    mbar_drain(drain, 0);
  }
  __syncwarp();
  // ---------------- epilogue: TMEM lane quarter -> logits rows ----------------
  const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, a.wait_cycles));
  tc_fence_after();
  if (ok) {
    const int v = v0 + 32 * warp + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    uint32_t r[32];
    for (int c0 = 0; c0 < a.Mp; c0 += 32) {
      tmem_ld32(lane_base + (uint32_t)c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int m = c0 + c;
        if (m < a.M && v < a.V) a.out[(long long)m * a.ldo + v] = __uint_as_float(r[c]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols) : "memory");
  }
  if (!ok && t == 0) flag_status(a.dev_status, ET_DEV_TIMEOUT);
}

bool make_map_rows(CUtensorMap *m, const void *base, long long rows, int H, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kLmK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace et

using namespace et;

extern "C" et_status et_lm_head(const et_lmhead_shape *s, const void *features, const void *weight, float *logits,
                                int32_t *dev_status, et_stream_t stream) {
  ET_RETURN_IF(!s || !features || !weight || !logits, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(s->M < 1 || s->M > kLmMaxN || s->H < kLmK || s->V < 1 || s->ldo < s->V, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(s->H % kLmK != 0 || s->V >= (1 << 30), ET_ERR_UNSUPPORTED);  // whole 64-element k slices
  ET_RETURN_IF(!et_aligned(features, 16) || !et_aligned(weight, 16) || !et_aligned(logits, 4), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!encode_fn(), ET_ERR_CUDA);
  const int Mp = s->M <= 16 ? 16 : (s->M <= 32 ? 32 : 64);
  const int stages = Mp <= 16 ? 6 : (Mp <= 32 ? 5 : 4);
  const size_t smem = (size_t)stages * (kLmABytes + (size_t)Mp * 128) + 8 * (2 * stages + 1) + 32 + 1024;
  CUtensorMap m_w, m_x;
  if (!make_map_rows(&m_w, weight, s->V, s->H, kLmRows) || !make_map_rows(&m_x, features, s->M, s->H, Mp))
    return ET_ERR_INVALID_ARG;
  if (et_smem_attr((const void *)k_lmhead_tc, kLmSmemMax) != cudaSuccess) return ET_ERR_CUDA;
  LmArgs a;
  a.M = s->M; a.Mp = Mp; a.H = s->H; a.V = s->V; a.stages = stages; a.ldo = s->ldo;
  a.out = logits;
  a.dev_status = dev_status;
  a.wait_cycles = et_wait_limit_cycles();
  return et_launch(k_lmhead_tc, dim3((s->V + kLmRows - 1) / kLmRows), dim3(kLmThreads), smem, (cudaStream_t)stream,
                   0, m_w, m_x, a);
}
