// Internal declarations shared by the libupf host code and its kernels.
//
// Work decomposition of the two scoring passes (UniPrefill article, section 二
// first step; section 三, scores + online normalisation):
//   * query rows of kv-group g: rho in [0, QR), QR = gamma * n; row rho is the
//     tail query j = rho % n of the q-head qhead[g*gamma + rho / n]; its
//     position in the request is t = L - n + j and it exists only if t >= 0.
//   * the rows of a group are cut into NQC chunks of QC rows;
//   * keys of request r are cut into splits of KS1 (pass 1) / KS2 (pass 2) keys;
//   * an item is (request r, kv head g, query chunk qc, key split s), numbered
//     request-major; item_off[r] is the first item of request r.
// Pass 1 writes per item and row the partial (m2, Z): m2 = max over the item's
// visible keys of x = scale*log2(e)*(q.k), Z = sum 2^(x - m2).  Pass 2 merges
// the partials of (r, g, qc) into lse2 = m2 + log2 Z and accumulates
// sum_rows 2^(x - lse2) per key into part[g*NQC + qc][token].
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "upf.h"

namespace upf {

constexpr int kMaxHeads = 256;         // H_q limit (the q-head list travels by value)
constexpr int kMaxBlocksPerReq = 16384;  // select kernel sorts up to this many blocks in shared memory
constexpr int kCompactChunkWords = 4096;  // keep-bit words per compaction chunk (131072 tokens)
constexpr int kPlanSMs = 152;             // SM count the work split is planned for (GB300)
// Partial rows the tensor-core passes write per (kv head, query chunk) and
// per pass-1 item row (the epilogue warps that split a unit's columns merge
// their sums inside the CTA).
constexpr int kTcPartials = 1;
// Longest a pipeline wait inside the tensor-core kernels may take by default,
// in SM clock cycles (about 2 s at 2 GHz).
constexpr long long kDefaultWaitCycles = 4000000000LL;

// Descriptor tables of a batch (cu_seqlens, the first item of each request in
// pass 1 and pass 2, the first block of each request), computed on the host
// from cu_seqlens_host.  The fused path carries them in the kernel parameters
// for batches of up to kInlineReqs requests, so no kernel has to build them on
// the device first; larger batches (and the separate entry points) keep them
// in the workspace, written by describe_kernel.
constexpr int kInlineReqs = 64;
struct DescInline {
  int32_t R;                     // 0: not carried (read the workspace tables)
  int32_t cu[kInlineReqs + 1];
  int32_t off1[kInlineReqs + 1];
  int32_t off2[kInlineReqs + 1];
  int32_t blk[kInlineReqs + 1];
};

// The tables one kernel reads, wherever they live.
struct DescView {
  const int32_t* cu;
  const int32_t* off1;
  const int32_t* off2;
  const int32_t* blk;
};

struct ScoreArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  int64_t q_stride;      // elements between consecutive tokens of q
  int64_t k_stride;      // elements between consecutive tokens of k
  const int32_t* cu;     // device cu_seqlens [R+1]
  int32_t R, T, Hq, Hkv, d, n, gamma;
  int32_t QR, QC, NQC;      // this pass's query chunks: NQC chunks of QC rows per group
  int32_t QC1, NQC1;        // pass 1's chunks (where pass 2 reads the pass-1 partials); QC is a multiple of QC1
  int32_t KS1, KS2;
  int32_t items1, items2;  // host totals (grid sizes)
  float scale_log2;
  int32_t q_box_rows;        // tail rows per TMA box of q (divides n)
  int32_t use_tc;            // 1: tcgen05 kernels, 0: CUDA-core kernels
  int32_t use_pair;          // 1: the tcgen05 kernels on CTA pairs (cta_group::2)
  const int32_t* item_off1;  // [R+1]
  const int32_t* item_off2;  // [R+1]
  float2* p1part;            // [items1][pw][QC]
  float* part;               // [Hkv*NQC*pw][T] (pass 2's NQC)
  int32_t pw;                // partial rows per item row / per (g, qc): kTcPartials or 1
  int32_t* status;
  long long wait_limit;      // pipeline waits of the tensor-core kernels (cycles)
  int32_t* counters;         // [ncounters] cleared by pass 1 for the tail kernel when
  int32_t ncounters;         //   desc.R > 0 (describe_kernel clears them otherwise)
  int32_t qhead[kMaxHeads];  // q heads of group g at [g*gamma, (g+1)*gamma)
  DescInline desc;           // desc.R > 0: these tables, and the device cu_seqlens only checked
};

struct DescribeArgs {
  const int32_t* cu;
  int32_t R, T, Hkv, NQC, NQC2, KS1, KS2, G;   // NQC, NQC2: query chunks per group of pass 1, pass 2
  int32_t items1, items2, NB;  // host totals: the device-derived ones must match
  int32_t* item_off1;
  int32_t* item_off2;
  int32_t* blk_off;
  int32_t* status;
  int32_t* counters;     // [ncounters] cleared here for the tail kernel (nullable)
  int32_t ncounters;
};

struct SelectArgs {
  const int32_t* cu;
  int32_t R, T, G, sink_keep, tail_keep, n;
  int32_t Hq;
  int32_t NB;             // total blocks (host value)
  int32_t max_nb;         // largest per-request block count (host value)
  int32_t P;              // partial rows in part (0 = read `scores`)
  float top_p;
  const float* part;      // [P][T] (fused path)
  const float* scores_in; // [T] (upf_select path)
  float* scores_out;      // [T] or null (fused path)
  float* block_scores;    // [NB]
  const int32_t* blk_off; // [R+1]
  uint32_t* keep_bits;    // [ceil(T/32)]
  int32_t* kept_count;    // [R]
  int32_t* status;
};

// The fused tail (finalize, block means, selection, keep bits, kept-token
// list, compacted offsets) of upf_select_tokens and upf_select.
constexpr int kTailMaxBpc = 32;   // blocks per CTA of the tail kernel (upper bound)
constexpr int kTailMaxBlock = 4096;  // larger G take the separate kernels

struct TailArgs {
  SelectArgs s;
  int32_t* counters;    // [R+1], zero on entry: CTAs done per request, then requests done
  uint32_t* edge_bits;  // [2R] keep bits of each request's first and last word when shared
  int32_t* kept_blk;    // [NB] (nullable): request r's kept blocks, in order, at blk_off[r] + m
  int32_t* kept_off;    // [NB]: output offset (within the request) of each of those blocks
  int32_t* kept_nblk;   // [R]: kept blocks per request
  int32_t* cu_out;      // [R+1] (nullable, then total_kept too)
  int32_t* total_kept;  // [1]
  int32_t nonempty;     // requests with at least one token (host value)
  int32_t bpc;          // blocks per CTA
  int32_t nbp;          // selection scratch capacity in blocks (multiple of 8, >= max_nb)
  DescInline desc;      // desc.R > 0: cu and block offsets from here, not s.cu / s.blk_off
};

struct CompactArgs {
  const int32_t* cu;
  int32_t R, T, nwords, nchunks;
  const uint32_t* keep_bits;
  int32_t* chunk_tot;     // [nchunks]
  int32_t* kept_index;    // [T]
  int64_t row_bytes;
  const void* hidden_in;
  void* hidden_out;
  const int64_t* pos_in;
  int64_t* pos_out;
  const int64_t* slot_in;
  int64_t* slot_out;
  int32_t* cu_out;
  int32_t* total_kept;
  int32_t layer_id, history_cap;
  int32_t* history;
  int32_t* history_len;
  int32_t* status;
};

struct ReviveArgs {
  int32_t T;
  const int32_t* kept_index;
  const int32_t* total_kept;
  const void* rows;
  void* full;
  int64_t row_bytes;
};

struct HistoryArgs {
  const int32_t* cu;
  int32_t R, layer_id, history_cap;
  const int32_t* history;
  const int32_t* history_len;
  int32_t* kv_len;
};

// Programmatic dependent launch.  Kernels launched after the first one of an
// API call may start while their predecessor is finishing; each kernel lets its
// own dependent start early and waits for its predecessor (full completion and
// memory visibility) before touching global memory.  Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Device status word helpers: the first error code wins.
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Sets the thread-local message returned by upf_last_error().
void set_last_error(const char* msg);

// Launchers (defined in the kernel translation units); all return cudaGetLastError().
cudaError_t launch_describe(const DescribeArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass1(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass2(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass1_tc(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass2_tc(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass1_pair(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_score_pass2_pair(const ScoreArgs& a, cudaStream_t s, bool pdl = false);
size_t score_pair_smem_bytes(int pass, int d, int QC);
constexpr int kPairTileKeys = 256;   // keys per tile of a CTA pair (key splits are multiples)
// Dynamic shared memory of a tensor-core pass (1 or 2) for head dim d and QC
// rows per query chunk, and its keys per tile (key splits are multiples of it).
size_t score_tc_smem_bytes(int pass, int d, int QC);
int score_tc_key_tile(int pass, int d);
cudaError_t launch_block_means(const SelectArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_compact_count(const CompactArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_compact_index(const CompactArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_compact_gather(const CompactArgs& a, cudaStream_t s, bool pdl = false);
int tail_blocks_per_cta(int G);
size_t tail_smem_bytes(int G, int max_nb);
cudaError_t launch_tail(const TailArgs& a, cudaStream_t s, bool pdl = false);
// The gather of the fused path, driven by the tail kernel's kept-block lists.
struct GatherListArgs {
  CompactArgs c;
  const int32_t* blk_off;   // [R+1]
  const int32_t* kept_blk;
  const int32_t* kept_off;
  const int32_t* kept_nblk;
  int32_t G;
  DescInline desc;          // desc.R > 0: cu and block offsets from here, not c.cu / blk_off
};
cudaError_t launch_gather_list(const GatherListArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_revive(const ReviveArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_history_kv_len(const HistoryArgs& a, cudaStream_t s, bool pdl = false);

}  // namespace upf
