// Cross-layer helpers around the selection path.
//
// Revival (UniPrefill article, section 二 third step): the hidden states of
// dropped tokens are frozen and carried forward; when a later layer needs the
// full-length sequence again, the rows the intermediate layers produced for the
// kept tokens are written back to their token positions and every dropped
// token keeps its frozen state.
//
// KV lengths from the drop history (section 三, last paragraph): decode reads
// the (layer id, kept count) records to know how many KV entries each layer
// wrote; a layer at or after a drop holds that drop's kept count until the next
// drop, and the prompt length before the first one.
#include "upf_internal.cuh"

namespace upf {

namespace {

// One warp per compacted row: full[kept_index[o]] = rows[o], 16-byte vectors.
__global__ void __launch_bounds__(256) revive_kernel(const ReviveArgs a) {
  pdl_trigger();
  pdl_wait();
  const int total = min(*a.total_kept, a.T);
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int64_t nvec = a.row_bytes / 16;
  for (int o = warp; o < total; o += nwarps) {
    const int t = a.kept_index[o];
    if (t < 0 || t >= a.T) continue;   // not a row of this batch: leave the buffer alone
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.rows) + (int64_t)o * a.row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.full) + (int64_t)t * a.row_bytes);
    int64_t v = lane;
    for (; v + 96 < nvec; v += 128) {
      const uint4 x0 = __ldcs(src + v), x1 = __ldcs(src + v + 32), x2 = __ldcs(src + v + 64), x3 = __ldcs(src + v + 96);
      __stcs(dst + v, x0);
      __stcs(dst + v + 32, x1);
      __stcs(dst + v + 64, x2);
      __stcs(dst + v + 96, x3);
    }
    for (; v < nvec; v += 32) __stcs(dst + v, __ldcs(src + v));
  }
}

// One thread per request: the kept count of its latest record at or before
// layer_id, else the request's prompt length.
__global__ void __launch_bounds__(256) history_kv_len_kernel(const HistoryArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= a.R) return;
  int kv = a.cu[r + 1] - a.cu[r];
  const int len = min(max(a.history_len[r], 0), a.history_cap);
  const int32_t* rec = a.history + (int64_t)r * a.history_cap * 2;
  for (int i = 0; i < len; ++i)
    if (rec[2 * i] <= a.layer_id) kv = rec[2 * i + 1];
  a.kv_len[r] = kv;
}

}  // namespace

cudaError_t launch_revive(const ReviveArgs& a, cudaStream_t s, bool pdl) {
  int blocks = (a.T + 7) / 8;
  blocks = blocks < 1 ? 1 : (blocks > 8 * kPlanSMs ? 8 * kPlanSMs : blocks);
  return launch_kernel(revive_kernel, blocks, 256, 0, s, pdl, a);
}

cudaError_t launch_history_kv_len(const HistoryArgs& a, cudaStream_t s, bool pdl) {
  const int blocks = (a.R + 255) / 256;
  return launch_kernel(history_kv_len_kernel, blocks < 1 ? 1 : blocks, 256, 0, s, pdl, a);
}

}  // namespace upf
