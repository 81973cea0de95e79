// upf_select_noalloc: upf_select (block means, top-p selection, exemption, keep
// mask) for callers that cannot allocate device memory.
//
// Who needs it: a serving engine that reserves nearly all of the GPU's memory
// for its own pools at start-up (KV cache, activations) and hands libraries no
// allocation hook, or a plugin that runs inside such an engine and may not go
// around the engine's allocator, cannot call cudaMalloc for a workspace at the
// point of the call and often cannot keep a library context around either.
// This entry point takes only its inputs and outputs: the scratch the select
// kernels need (the batch descriptor and, when the caller passes no
// block_scores buffer, the block means) lives in one file-scope device array
// of fixed size, compiled into the library.
//
// That array is shared by every call in the process on a given GPU and keeps
// the last call's contents; each call rewrites all of it that it reads, and
// clears the status word it may use.  Calls whose GPU work overlaps (two
// streams, or two host threads) race on it and must be serialised by the
// caller.  Every GPU on which the library's code is loaded holds the array
// until the process exits.
#include <mutex>

#include "upf_internal.cuh"

namespace {

constexpr int kMaxReqs = UPF_NOALLOC_MAX_REQS;
constexpr int kMaxBlocks = UPF_NOALLOC_MAX_BLOCKS;
constexpr size_t kStatusBytes = 256;
constexpr size_t kDescBytes = ((sizeof(int32_t) * 3 * (kMaxReqs + 1)) + 255) & ~size_t(255);
constexpr size_t kBlockBytes = sizeof(float) * kMaxBlocks;
constexpr size_t kScratchBytes = kStatusBytes + kDescBytes + kBlockBytes;

// The scratch: [status word | descriptor | block means].
static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_dev[kMaxDevices] = {};

upf_status reject(upf_status code, const char* msg) {
  upf::set_last_error(msg);
  return code;
}

// Device address of the scratch array on the current device.  The host-side
// name g_select_scratch is only a stand-in, never a device address; the real
// address comes from cudaGetSymbolAddress, once per device, with that device
// current.
upf_status scratch_address(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return reject(UPF_ERR_CUDA, "upf_select_noalloc: no usable current device");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess || !p) return reject(UPF_ERR_CUDA, "upf_select_noalloc: cudaGetSymbolAddress failed");
    g_scratch_dev[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_dev[dev];
  return UPF_OK;
}

}  // namespace

extern "C" upf_status upf_select_noalloc(const upf_batch* batch, const upf_params* params, const float* scores,
                                         float* block_scores, uint32_t* keep_bits, int32_t* kept_count,
                                         int32_t* status_dev, void* stream) {
  if (!batch || !params) return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: batch and params are required");
  if (!scores || !keep_bits || !kept_count)
    return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: scores, keep_bits and kept_count are required");
  const int R = batch->num_reqs;
  if (R < 1) return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: num_reqs must be >= 1");
  if (R > kMaxReqs)
    return reject(UPF_ERR_UNSUPPORTED, "upf_select_noalloc: more than UPF_NOALLOC_MAX_REQS (1024) requests");
  const int32_t* cu = batch->cu_seqlens_host;
  if (!cu || !batch->cu_seqlens_dev) return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: cu_seqlens are required");
  if (cu[0] != 0) return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: cu_seqlens[0] must be 0");
  if (params->block < 1 || params->block > (1 << 20))
    return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: block must be in [1, 2^20]");
  if (!(params->top_p > 0.f && params->top_p <= 1.f))
    return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: top_p must be in (0, 1]");
  if (params->sink_keep < 0 || params->tail_keep < 0)
    return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: sink_keep/tail_keep must be >= 0");
  long long nb_total = 0;
  int max_nb = 0, nonempty = 0;
  for (int r = 0; r < R; ++r) {
    const int L = cu[r + 1] - cu[r];
    if (L < 0) return reject(UPF_ERR_INVALID_ARG, "upf_select_noalloc: cu_seqlens must be non-decreasing");
    const int nb = int((L + (long long)params->block - 1) / params->block);
    nb_total += nb;
    max_nb = nb > max_nb ? nb : max_nb;
    nonempty += L > 0;
  }
  if (cu[R] > (1 << 30)) return reject(UPF_ERR_UNSUPPORTED, "upf_select_noalloc: total tokens above 2^30");
  if (nb_total > kMaxBlocks)
    return reject(UPF_ERR_UNSUPPORTED, "upf_select_noalloc: more than UPF_NOALLOC_MAX_BLOCKS (65536) blocks");
  if (max_nb > upf::kMaxBlocksPerReq)
    return reject(UPF_ERR_UNSUPPORTED, "upf_select_noalloc: a request has more than 16384 blocks");

  unsigned char* base = nullptr;
  upf_status st = scratch_address(&base);
  if (st != UPF_OK) return st;
  int32_t* own_status = reinterpret_cast<int32_t*>(base);
  int32_t* desc = reinterpret_cast<int32_t*>(base + kStatusBytes);
  float* bs_scratch = reinterpret_cast<float*>(base + kStatusBytes + kDescBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = status_dev ? status_dev : own_status;
  if (!status_dev) {
    cudaError_t e = cudaMemsetAsync(own_status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return reject(UPF_ERR_CUDA, "upf_select_noalloc: clearing the status word failed");
  }

  // Batch descriptor.  Only the block offsets are used here; the two item
  // tables are sized to one item per non-empty request.
  upf::DescribeArgs da;
  da.cu = batch->cu_seqlens_dev;
  da.R = R;
  da.T = cu[R];
  da.Hkv = 1;
  da.NQC = da.NQC2 = 1;
  da.KS1 = da.KS2 = 1 << 30;
  da.G = params->block;
  da.items1 = da.items2 = nonempty;
  da.NB = int(nb_total);
  da.item_off1 = desc;
  da.item_off2 = desc + (R + 1);
  da.blk_off = desc + 2 * (R + 1);
  da.status = status;
  da.counters = nullptr;
  da.ncounters = 0;
  cudaError_t e = upf::launch_describe(da, s);
  if (e != cudaSuccess) return reject(UPF_ERR_CUDA, "upf_select_noalloc: describe launch failed");

  upf::SelectArgs sa;
  sa.cu = batch->cu_seqlens_dev;
  sa.R = R;
  sa.T = cu[R];
  sa.G = params->block;
  sa.sink_keep = params->sink_keep;
  sa.tail_keep = params->tail_keep;
  sa.n = params->n_tail > 0 ? params->n_tail : 1;
  sa.Hq = batch->num_q_heads > 0 ? batch->num_q_heads : 1;
  sa.NB = int(nb_total);
  sa.max_nb = max_nb;
  sa.P = 0;
  sa.top_p = params->top_p;
  sa.part = nullptr;
  sa.scores_in = scores;
  sa.scores_out = nullptr;
  sa.block_scores = block_scores ? block_scores : bs_scratch;
  sa.blk_off = da.blk_off;
  sa.keep_bits = keep_bits;
  sa.kept_count = kept_count;
  sa.status = status;
  if ((e = upf::launch_block_means(sa, s)) != cudaSuccess)
    return reject(UPF_ERR_CUDA, "upf_select_noalloc: block-means launch failed");
  if ((e = upf::launch_select(sa, s)) != cudaSuccess) return reject(UPF_ERR_CUDA, "upf_select_noalloc: select launch failed");
  return UPF_OK;
}
