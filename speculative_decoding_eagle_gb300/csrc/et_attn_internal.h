// Internal interface between the attention entry point (et_attention.cu) and
// the tcgen05 kernel (et_attention_tc.cu).  Not part of the C ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "eagle_tree.h"

#define ET_HIDDEN __attribute__((visibility("hidden")))

namespace et {

struct TcLaunch {
  int B, N, Hq, Hkv, G, MT, S, W;  // MT row tiles of 128 per KV head, S KV splits
  float scale_log2;
  const void *q, *kp, *vp, *kt, *vt;
  const long long *kv_row0;
  const int *prefix_len;
  long long kv_rows, kv_head_stride;
  const unsigned long long *mask;
  void *out;
  float *lse;
  int *dev_status;
  float *ws;   // S > 1: partial rows [B*Hkv*MT][S][128][128], then (max, sum) [B*Hkv*MT][S][128]
  int q_tma;   // set by the launcher: the Q tile comes by TMA (G divides 128)
  long long wait_cycles;  // bound of every mbarrier wait (et_set_wait_limit)
  int inputs_ready;       // ET_ATTN_INPUTS_READY: the first tiles may be fetched before the programmatic wait
};

constexpr int kTcRows = 128;   // query rows per tile (TMEM lanes)
constexpr int kTcKeys = 64;    // keys per K/V tile
constexpr int kTcDim = 128;    // head dim of the tcgen05 path
constexpr int kTcMaxSplits = 16;  // KV splits of one row tile = one thread-block cluster (past 8: non-portable size)
constexpr int kLptMaxB = 64;      // batches whose sequences go out longest prefix first (tcgen05 path)

// workspace bytes of the tcgen05 path: the split merge's partial rows and
// (max, sum) pairs (0 for one split)
inline size_t tc_workspace_bytes(long long tiles, int S) {
  return S > 1 ? (size_t)tiles * S * kTcRows * (kTcDim * 4 + 8) : 0;
}

ET_HIDDEN et_status tc_attention_launch(const TcLaunch &a, cudaStream_t stream);

}  // namespace et
