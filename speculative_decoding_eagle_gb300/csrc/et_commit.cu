// KV commit after acceptance (EAGLE-2 article on sbmmt.com, reranking phase
// and attention mask: row 0 of the flattened tree is the root, every row
// attends the prefix plus its ancestors; EAGLE blog section 1.1: the accepted
// tokens of one verification forward are kept).  The root row and the
// accepted draft rows path[1..accept_len] are appended to the KV cache in
// path order at positions prefix_len.., their features gathered for the next
// draft step, and the prefix length advanced by accept_len + 1.
//
// One block per (path position, sequence); each copies Hkv K rows, Hkv V
// rows and one feature row with 16-byte vector loads and stores.  The bytes
// are few ((D+1) x Hkv x d per sequence), so the kernel is latency-bound; it
// exists so that the step never leaves the device between acceptance and the
// next draft.
#include "et_common.cuh"

namespace et {
namespace {

constexpr int kCmThreads = 256;

struct CommitArgs {
  int B, N, Hkv, path_len, chunks_kv, chunks_f;  // 16-byte chunks per head row / feature row
  long long head_stride, kv_rows, feat_chunks_row;
  const uint4 *k_tree, *v_tree, *features;
  const int32_t *accept_len, *path, *prefix_len;
  const long long *kv_row0;
  uint4 *k_cache, *v_cache, *feat_out;
  int32_t *new_prefix_len, *dev_status;
};

__global__ void __launch_bounds__(kCmThreads) k_kv_commit(CommitArgs a) {
  pdl_wait();     // the previous kernel in the stream has completed
  pdl_trigger();  // only now may the next kernel launch: at most one waits ahead
  const int i = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int alen = a.accept_len[b];
  const bool alen_ok = alen >= 0 && alen < a.path_len;
  if (i == 0 && t == 0) {
    if (alen_ok) a.new_prefix_len[b] = a.prefix_len[b] + alen + 1;
    else flag_status(a.dev_status, ET_DEV_BAD_INDEX);
  }
  if (!alen_ok || i > alen) {  // past the accepted path: zero feature row
    if (a.feat_out)
      for (int c = t; c < a.chunks_f; c += kCmThreads)
        a.feat_out[((long long)b * a.path_len + i) * a.chunks_f + c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int row = a.path[(long long)b * a.path_len + i];
  const long long pos = (long long)a.prefix_len[b] + i;
  const long long base = a.kv_row0[b];
  const bool ok = row >= 0 && row < a.N && pos >= 0 && pos < a.head_stride && base >= 0 &&
                  base + (a.Hkv - 1) * a.head_stride + pos < a.kv_rows;
  if (!ok) {
    if (t == 0) flag_status(a.dev_status, ET_DEV_BAD_INDEX);
    return;
  }
  const int per_head = a.chunks_kv;
  const long long src0 = ((long long)b * a.N + row) * a.Hkv * per_head;
  for (int c = t; c < a.Hkv * per_head; c += kCmThreads) {
    const int g = c / per_head, x = c - g * per_head;
    const long long dst = (base + g * a.head_stride + pos) * per_head + x;
    a.k_cache[dst] = a.k_tree[src0 + c];
    a.v_cache[dst] = a.v_tree[src0 + c];
  }
  if (a.feat_out && a.features)
    for (int c = t; c < a.chunks_f; c += kCmThreads)
      a.feat_out[((long long)b * a.path_len + i) * a.chunks_f + c] =
          a.features[((long long)b * a.N + row) * a.chunks_f + c];
}

}  // namespace
}  // namespace et

using namespace et;

extern "C" et_status et_kv_commit(const et_commit_shape *s, const void *k_tree, const void *v_tree,
                                  const int32_t *accept_len, const int32_t *path, void *k_cache, void *v_cache,
                                  const int64_t *kv_row0, const int32_t *prefix_len, int32_t *new_prefix_len,
                                  const void *features, void *feat_out, int32_t *dev_status, et_stream_t stream) {
  ET_RETURN_IF(!s, ET_ERR_INVALID_ARG);
  ET_RETURN_IF(s->dtype != ET_BF16 && s->dtype != ET_F32, ET_ERR_INVALID_ARG);
  const int es = s->dtype == ET_BF16 ? 2 : 4;
  ET_RETURN_IF(s->B < 1 || s->B > 65535 || s->N < 1 || s->N > kMaxN || s->Hkv < 1 || s->d < 1 ||
                   s->path_len < 1 || s->path_len > kMaxDepth + 1 || s->kv_head_stride < 1 || s->kv_rows < 1 ||
                   s->feat_dim < 0,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(((long long)s->d * es) % 16 != 0 || ((long long)s->feat_dim * es) % 16 != 0, ET_ERR_UNSUPPORTED);
  ET_RETURN_IF(!k_tree || !v_tree || !accept_len || !path || !k_cache || !v_cache || !kv_row0 || !prefix_len ||
                   !new_prefix_len,
               ET_ERR_INVALID_ARG);
  ET_RETURN_IF(new_prefix_len == prefix_len, ET_ERR_INVALID_ARG);  // blocks of a sequence read prefix_len
  ET_RETURN_IF(s->feat_dim > 0 && (!features || !feat_out), ET_ERR_INVALID_ARG);
  ET_RETURN_IF(!et_aligned(k_tree, 16) || !et_aligned(v_tree, 16) || !et_aligned(k_cache, 16) ||
                   !et_aligned(v_cache, 16) || (features && !et_aligned(features, 16)) ||
                   (feat_out && !et_aligned(feat_out, 16)),
               ET_ERR_INVALID_ARG);
  CommitArgs a;
  a.B = s->B; a.N = s->N; a.Hkv = s->Hkv; a.path_len = s->path_len;
  a.chunks_kv = (int)((long long)s->d * es / 16);
  a.chunks_f = (int)((long long)s->feat_dim * es / 16);
  a.head_stride = s->kv_head_stride;
  a.kv_rows = s->kv_rows;
  a.feat_chunks_row = a.chunks_f;
  a.k_tree = static_cast<const uint4 *>(k_tree);
  a.v_tree = static_cast<const uint4 *>(v_tree);
  a.features = s->feat_dim > 0 ? static_cast<const uint4 *>(features) : nullptr;
  a.accept_len = accept_len; a.path = path; a.prefix_len = prefix_len;
  a.kv_row0 = reinterpret_cast<const long long *>(kv_row0);
  a.k_cache = static_cast<uint4 *>(k_cache);
  a.v_cache = static_cast<uint4 *>(v_cache);
  a.feat_out = s->feat_dim > 0 ? static_cast<uint4 *>(feat_out) : nullptr;
  a.new_prefix_len = new_prefix_len;
  a.dev_status = dev_status;
  return et_launch(k_kv_commit, dim3(s->path_len, s->B), dim3(kCmThreads), 0, (cudaStream_t)stream, 0, a);
}
