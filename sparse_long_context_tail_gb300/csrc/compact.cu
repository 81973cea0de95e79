// Compaction of kept tokens and the drop-history append.
//
// UniPrefill article, section 二 third step: after the drop every later layer
// runs on the kept tokens only, and the dropped tokens' hidden states stay
// frozen (here: untouched in the input buffers); section 三: the batch metadata
// (positions, KV-cache slot addresses) follows the drop, and each drop records
// the layer id and the number of kept tokens.
//
// Three launches: (1) popcount per chunk of 4096 keep-bit words (skipped when
// the batch fits one chunk, up to 131072 tokens); (2) per chunk, a block scan of
// word popcounts gives every kept token its output row, written to kept_index,
// plus the compacted cu_seqlens of the requests that start in the chunk; (3) a
// persistent gather, one warp per output row, moving hidden rows with 16-byte
// vector loads/stores, plus the history append.
#include "upf_internal.cuh"

namespace upf {

namespace {

constexpr int kChunkThreads = 1024;

// Keep-bit word w with any bits past token T cleared (defensive: a caller's
// mask may carry stray bits there, which must not produce rows past T).
__device__ __forceinline__ uint32_t load_word(const CompactArgs& a, int w) {
  if (w >= a.nwords) return 0u;
  uint32_t x = a.keep_bits[w];
  if (w == a.nwords - 1 && (a.T & 31)) x &= (1u << (a.T & 31)) - 1u;
  return x;
}
constexpr int kWordsPerThread = kCompactChunkWords / kChunkThreads;  // 4
static_assert(kWordsPerThread * kChunkThreads == kCompactChunkWords, "a chunk is split evenly");

__device__ __forceinline__ int block_sum(int v, int* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_tmp[warp] = v;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_tmp[w];
  __syncthreads();
  return tot;
}

__global__ void __launch_bounds__(kChunkThreads) compact_count_kernel(const CompactArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_tmp[kChunkThreads / 32];
  const int c = blockIdx.x;
  int cnt = 0;
  for (int i = 0; i < kWordsPerThread; ++i) {
    const int w = c * kCompactChunkWords + threadIdx.x * kWordsPerThread + i;
    cnt += __popc(load_word(a, w));
  }
  const int tot = block_sum(cnt, s_tmp);
  if (threadIdx.x == 0) a.chunk_tot[c] = tot;
}

__global__ void __launch_bounds__(kChunkThreads) compact_index_kernel(const CompactArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_tmp[kChunkThreads / 32];
  __shared__ int s_woff[kCompactChunkWords + 1];  // exclusive kept-token prefix per word of the chunk
  __shared__ uint32_t s_word[kCompactChunkWords];
  __shared__ int s_warp[kChunkThreads / 32];
  const int c = blockIdx.x, tid = threadIdx.x;
  // Kept tokens in earlier chunks.
  int before = 0;
  for (int i = tid; i < c; i += blockDim.x) before += a.chunk_tot[i];
  const int base = block_sum(before, s_tmp);
  // Word popcounts and their exclusive scan within the chunk.
  uint32_t words[kWordsPerThread];
  int pc[kWordsPerThread];
  int mine = 0;
  for (int i = 0; i < kWordsPerThread; ++i) {
    const int w = c * kCompactChunkWords + tid * kWordsPerThread + i;
    words[i] = load_word(a, w);
    pc[i] = __popc(words[i]);
    mine += pc[i];
  }
  const int lane = tid & 31, warp = tid >> 5;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int woff = 0;
  for (int w = 0; w < warp; ++w) woff += s_warp[w];
  int run = woff + incl - mine;
  for (int i = 0; i < kWordsPerThread; ++i) {
    s_woff[tid * kWordsPerThread + i] = run;
    s_word[tid * kWordsPerThread + i] = words[i];
    run += pc[i];
  }
  if (tid == blockDim.x - 1) s_woff[kCompactChunkWords] = run;
  __syncthreads();
  // Output rows: one word per warp at a time, lane b writing the row of bit
  // b, so each warp's stores are consecutive.
  for (int wl = warp; wl < kCompactChunkWords; wl += kChunkThreads / 32) {
    const uint32_t word = s_word[wl];
    if ((word >> lane) & 1u)
      a.kept_index[base + s_woff[wl] + __popc(word & ((1u << lane) - 1u))] =
          (c * kCompactChunkWords + wl) * 32 + lane;
  }
  // Compacted cu_seqlens: boundary r lies in this chunk if its first token
  // does; the last chunk also takes every boundary at or past its start
  // (including cu[R] = T).
  const int tok_lo = c * kCompactChunkWords * 32;
  const int tok_hi = (c == a.nchunks - 1) ? 0x7fffffff : tok_lo + kCompactChunkWords * 32;
  for (int r = tid; r <= a.R; r += blockDim.x) {
    int t = a.cu[r];
    t = t < 0 ? 0 : (t > a.T ? a.T : t);
    if (t >= tok_lo && t < tok_hi) {
      const int lw = (t - tok_lo) >> 5;
      int v;
      if (lw >= kCompactChunkWords) {
        v = s_woff[kCompactChunkWords];
      } else {
        const int w = (t >> 5);
        const uint32_t word = load_word(a, w);
        const uint32_t below = (t & 31) ? (word & ((1u << (t & 31)) - 1u)) : 0u;
        v = s_woff[lw] + __popc(below);
      }
      a.cu_out[r] = base + v;
    }
  }
  if (c == a.nchunks - 1 && tid == 0) *a.total_kept = base + s_woff[kCompactChunkWords];
}

__global__ void __launch_bounds__(256) compact_gather_kernel(const CompactArgs a) {
  pdl_trigger();
  pdl_wait();
  const int total = min(*a.total_kept, a.T);
  // Drop history: one record per request, all or nothing.
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.history) {
    bool full = false;
    for (int r = 0; r < a.R; ++r) full |= a.history_len[r] >= a.history_cap || a.history_len[r] < 0;
    if (full) {
      set_status(a.status, UPF_ERR_CAPACITY);
    } else {
      for (int r = 0; r < a.R; ++r) {
        const int len = a.history_len[r];
        int32_t* rec = a.history + ((int64_t)r * a.history_cap + len) * 2;
        rec[0] = a.layer_id;
        rec[1] = a.cu_out[r + 1] - a.cu_out[r];
        a.history_len[r] = len + 1;
      }
    }
  }
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int64_t nvec = a.row_bytes / 16;
  for (int o = warp; o < total; o += nwarps) {
    const int t = a.kept_index[o];
    if (a.hidden_in) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.hidden_in) + (int64_t)t * a.row_bytes);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.hidden_out) + (int64_t)o * a.row_bytes);
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
    if (lane == 0 && a.pos_in) a.pos_out[o] = a.pos_in[t];
    if (lane == 1 && a.slot_in) a.slot_out[o] = a.slot_in[t];
  }
}

}  // namespace

cudaError_t launch_compact_count(const CompactArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(compact_count_kernel, a.nchunks, kChunkThreads, 0, s, pdl, a);
}

cudaError_t launch_compact_index(const CompactArgs& a, cudaStream_t s, bool pdl) {
  return launch_kernel(compact_index_kernel, a.nchunks, kChunkThreads, 0, s, pdl, a);
}

cudaError_t launch_compact_gather(const CompactArgs& a, cudaStream_t s, bool pdl) {
  // Enough warps to cover every row in one pass when few rows survive, capped
  // at a few waves of resident warps.
  int blocks = (a.T + 7) / 8;
  blocks = blocks < 1 ? 1 : blocks;
  blocks = blocks > 8 * kPlanSMs ? 8 * kPlanSMs : blocks;
  return launch_kernel(compact_gather_kernel, blocks, 256, 0, s, pdl, a);
}

}  // namespace upf
