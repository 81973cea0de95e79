// libupf host side: argument checks, work planning, workspace layout and the
// launch sequence of each C-ABI entry point declared in include/upf.h.
//
// Nothing here allocates except upf_create (one small device status word).
// Every launch goes to the caller's stream; argument errors are reported before
// the first launch.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "upf_internal.cuh"

struct upf_ctx {
  int device;
  int num_sms;
  int32_t* status_dev;  // [64] device words; [0] = status
  long long wait_limit = 0;  // pipeline waits of the scoring kernels, cycles (0: default)
  // tracing
  bool profiling = false;
  int32_t launches[UPF_NUM_STAGES] = {};
  struct Rec {
    int stage;
    cudaEvent_t a, b;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;

  cudaEvent_t event() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};

namespace {

thread_local std::string g_last_error;

upf_status fail(upf_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

upf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(UPF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Everything the launches need that follows from the batch and parameters.
struct Plan {
  int R = 0, T = 0, Hq = 0, Hkv = 0, d = 0, gamma = 0;
  int n = 0, G = 0, sink = 0, tail = 0;
  float top_p = 0.f, scale = 0.f;
  int QR = 0, QC = 0, NQC = 0, KS1 = 0, KS2 = 0;
  int QC2 = 0, NQC2 = 0;   // pass 2's query chunks (QC2 a multiple of QC)
  int pw = 1;   // partial rows per pass-1 item row and per (kv head, query chunk)
  int q_box_rows = 0;
  bool use_tc = false;
  bool use_pair = false;    // pass 1 on CTA pairs
  bool use_pair2 = false;   // pass 2 on CTA pairs
  long long items1 = 0, items2 = 0;
  long long NB = 0;
  int max_nb = 0;
  int nwords = 0, nchunks = 0;
  std::vector<int32_t> qhead;
  // workspace offsets
  size_t off_desc = 0, off_p1 = 0, off_part = 0, off_bs = 0, off_chunk = 0, off_kidx = 0, off_ctr = 0, off_kbl = 0,
         total = 0;
  int nonempty = 0;
};

// The fused tail kernel serves blocks up to kTailMaxBlock tokens; larger
// blocks take the separate finalize, select and compaction kernels.
bool fused_tail(const Plan& pl) { return pl.G >= 1 && pl.G <= upf::kTailMaxBlock; }

upf_status check_batch(const upf_batch* b) {
  if (!b) return fail(UPF_ERR_INVALID_ARG, "batch is NULL");
  if (b->num_reqs < 1) return fail(UPF_ERR_INVALID_ARG, "num_reqs must be >= 1 (got %d)", b->num_reqs);
  if (!b->cu_seqlens_host || !b->cu_seqlens_dev)
    return fail(UPF_ERR_INVALID_ARG, "cu_seqlens_host and cu_seqlens_dev are required");
  if (b->cu_seqlens_host[0] != 0) return fail(UPF_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
  for (int r = 0; r < b->num_reqs; ++r)
    if (b->cu_seqlens_host[r + 1] < b->cu_seqlens_host[r])
      return fail(UPF_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing (r=%d)", r);
  if (b->cu_seqlens_host[b->num_reqs] > (1 << 30))
    return fail(UPF_ERR_UNSUPPORTED, "total tokens %d above 2^30", b->cu_seqlens_host[b->num_reqs]);
  return UPF_OK;
}

upf_status check_heads(const upf_batch* b) {
  if (b->num_q_heads < 1 || b->num_kv_heads < 1 || b->num_q_heads % b->num_kv_heads != 0)
    return fail(UPF_ERR_INVALID_ARG, "need H_q %% H_kv == 0 and both >= 1 (got %d, %d)", b->num_q_heads,
                b->num_kv_heads);
  if (b->num_q_heads > upf::kMaxHeads)
    return fail(UPF_ERR_UNSUPPORTED, "num_q_heads %d above %d", b->num_q_heads, upf::kMaxHeads);
  if (b->head_dim != 64 && b->head_dim != 128 && b->head_dim != 256)
    return fail(UPF_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", b->head_dim);
  if (b->kv_of_q) {
    const int gamma = b->num_q_heads / b->num_kv_heads;
    std::vector<int> cnt(b->num_kv_heads, 0);
    for (int h = 0; h < b->num_q_heads; ++h) {
      int g = b->kv_of_q[h];
      if (g < 0 || g >= b->num_kv_heads) return fail(UPF_ERR_INVALID_ARG, "kv_of_q[%d]=%d out of range", h, g);
      cnt[g]++;
    }
    for (int g = 0; g < b->num_kv_heads; ++g)
      if (cnt[g] != gamma)
        return fail(UPF_ERR_INVALID_ARG, "kv_of_q maps %d q heads to kv head %d, need %d", cnt[g], g, gamma);
  }
  return UPF_OK;
}

upf_status check_params(const upf_params* p) {
  if (!p) return fail(UPF_ERR_INVALID_ARG, "params is NULL");
  if (p->n_tail < 1 || p->n_tail > 4096) return fail(UPF_ERR_UNSUPPORTED, "n_tail must be in [1, 4096]");
  if (p->block < 1 || p->block > (1 << 20)) return fail(UPF_ERR_INVALID_ARG, "block must be in [1, 2^20]");
  if (p->sink_keep < 0 || p->tail_keep < 0) return fail(UPF_ERR_INVALID_ARG, "sink_keep/tail_keep must be >= 0");
  if (!(p->top_p > 0.f && p->top_p <= 1.f)) return fail(UPF_ERR_INVALID_ARG, "top_p must be in (0, 1]");
  if (!std::isfinite(p->softmax_scale)) return fail(UPF_ERR_INVALID_ARG, "softmax_scale must be finite");
  return UPF_OK;
}

int ceil_div(long long a, long long b) { return int((a + b - 1) / b); }

// Keys per split so that the pass has about `target` items in total: a
// multiple of `tile` keys, at least 256 (the CUDA-core kernels, a few waves).
int choose_split(const upf_batch* b, int per_req_units, long long target, int tile) {
  long long keys = 0;
  for (int r = 0; r < b->num_reqs; ++r) keys += b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r];
  long long units = keys * per_req_units;
  long long ks = (units + target - 1) / std::max(1LL, target);
  ks = ((ks + tile - 1) / tile) * tile;
  if (ks < 256) ks = 256;
  return int(std::min<long long>(ks, 1 << 30));
}

long long split_items(const upf_batch* b, int units, long long ks) {
  long long n = 0;
  for (int r = 0; r < b->num_reqs; ++r) n += (long long)units * ceil_div(b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r], ks);
  return n;
}

// Estimated duration of a tensor-core pass with key splits of ks keys: the
// items, in launch order (request, kv head, split, query chunk), go to the
// first SM that is free (one CTA per SM); an item costs its keys plus a
// fixed start-up of `ovh` keys (query chunk load, tensor memory, pipeline
// fill and drain).
long long split_makespan(const upf_batch* b, int hkv, int nqc, long long ks, long long ovh, int sms) {
  std::vector<long long> heap(size_t(sms), 0);   // min-heap of SM finish times
  auto push_pop = [&](long long cost) {
    long long t = heap[0] + cost;
    size_t i = 0;   // replace the root and sift down
    for (;;) {
      size_t l = 2 * i + 1, r = l + 1, m = i;
      long long tm = t;
      if (l < heap.size() && heap[l] < tm) { m = l; tm = heap[l]; }
      if (r < heap.size() && heap[r] < tm) { m = r; tm = heap[r]; }
      if (m == i) break;
      heap[i] = heap[m];
      i = m;
    }
    heap[i] = t;
  };
  for (int r = 0; r < b->num_reqs; ++r) {
    const long long L = b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r];
    const long long nsplit = (L + ks - 1) / ks;
    for (int g = 0; g < hkv; ++g)
      for (long long sp = 0; sp < nsplit; ++sp)
        for (int qc = 0; qc < nqc; ++qc) push_pop(std::min(ks, L - sp * ks) + ovh);
  }
  return *std::max_element(heap.begin(), heap.end());
}

// Key splits of the tensor-core passes (one CTA per SM, one item per CTA).
// Rounding the ideal split up to whole tiles can leave a few items over a
// whole wave (160 items on 152 SMs take two item-times), so the split is
// chosen among the smallest splits that fit the items into 1..4 waves, by
// the estimated duration of each.
int choose_split_tc(const upf_batch* b, int hkv, int nqc, int tile, int sms) {
  const int units = hkv * nqc;
  long long keys = 0, max_len = 0;
  for (int r = 0; r < b->num_reqs; ++r) {
    const long long L = b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r];
    keys += L;
    max_len = std::max(max_len, L);
  }
  auto round_tile = [&](long long x) { return std::max<long long>(256, ((x + tile - 1) / tile) * tile); };
  const long long hi_ks = round_tile(std::max<long long>(max_len, 1));
  long long best = round_tile((keys * units + sms - 1) / sms);
  if (best > hi_ks) best = hi_ks;
  const long long n_best = split_items(b, units, best);
  // One wave already: no smaller split fits one wave, and more waves only add start-ups.
  if (n_best <= sms || n_best > (1LL << 20)) return int(std::min<long long>(best, 1 << 30));
  // The simulation below costs host time; batches repeat across layers and steps.
  struct Entry {
    uint64_t key = 0;
    int ks = 0;
  };
  thread_local Entry cache[8];
  thread_local int cache_next = 0;
  uint64_t key = 1469598103934665603ULL;
  auto mix = [&](uint64_t v) { key = (key ^ v) * 1099511628211ULL; };
  mix(uint64_t(b->num_reqs));
  mix(uint64_t(hkv));
  mix(uint64_t(nqc));
  mix(uint64_t(tile));
  mix(uint64_t(sms));
  for (int r = 0; r <= b->num_reqs; ++r) mix(uint64_t(uint32_t(b->cu_seqlens_host[r])));
  for (const Entry& e : cache)
    if (e.ks && e.key == key) return e.ks;
  const long long ovh = 2LL * tile;
  long long best_t = split_makespan(b, hkv, nqc, best, ovh, sms);
  // a geometric sweep around the ideal split (uneven request lengths make
  // the best split hard to predict) ...
  const long long ideal = (keys * units + sms - 1) / sms;
  for (int i = 0; i < 25; ++i) {
    // 1/8 x .. 2 x in steps of 2^(1/6)
    const long long ks = std::min(hi_ks, round_tile((long long)(double(ideal) * std::exp2(i / 6.0 - 3.0))));
    const long long t = split_makespan(b, hkv, nqc, ks, ovh, sms);
    if (t < best_t || (t == best_t && ks > best)) {
      best_t = t;
      best = ks;
    }
  }
  // ... and the smallest splits that fit the items into 1..4 waves
  for (int w = 1; w <= 4; ++w) {
    // smallest whole-tile split with at most w * sms items (items fall as the split grows)
    long long lo = round_tile((keys * units + (long long)w * sms - 1) / ((long long)w * sms)), hi = hi_ks;
    if (lo > hi) lo = hi;
    while (lo < hi) {
      const long long mid = round_tile(lo + (hi - lo) / 2);
      if (mid >= hi) break;
      if (split_items(b, units, mid) <= (long long)w * sms) hi = mid;
      else lo = mid + tile;
    }
    const long long ks = split_items(b, units, lo) <= (long long)w * sms ? lo : hi;
    const long long t = split_makespan(b, hkv, nqc, ks, ovh, sms);
    if (t < best_t || (t == best_t && ks > best)) {
      best_t = t;
      best = ks;
    }
  }
  const int chosen = int(std::min<long long>(best, 1 << 30));
  cache[cache_next] = Entry{key, chosen};
  cache_next = (cache_next + 1) % 8;
  return chosen;
}

upf_status make_plan(const upf_ctx* ctx, const upf_batch* b, const upf_params* p, bool need_heads, Plan* pl) {
  upf_status st = check_batch(b);
  if (st != UPF_OK) return st;
  if (need_heads) {
    if ((st = check_heads(b)) != UPF_OK) return st;
    if ((st = check_params(p)) != UPF_OK) return st;
  }
  pl->R = b->num_reqs;
  pl->T = b->cu_seqlens_host[b->num_reqs];
  if (need_heads) {
    pl->Hq = b->num_q_heads;
    pl->Hkv = b->num_kv_heads;
    pl->d = b->head_dim;
    pl->gamma = pl->Hq / pl->Hkv;
    pl->n = p->n_tail;
    pl->G = p->block;
    pl->sink = p->sink_keep;
    pl->tail = p->tail_keep;
    pl->top_p = p->top_p;
    pl->scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt(float(b->head_dim));
    pl->QR = pl->gamma * pl->n;
    // Query rows per chunk: the whole group's tail rows when they fit the
    // tensor-core kernels' shared-memory budget (512 rows of d <= 128, 256 rows
    // of d = 256), rounded up to whole 128-row MMA tiles.
    // At d = 256 a group of at most 256 rows is bound by the key reads (about
    // QR flop per key byte, below the tensor/HBM ridge): chunks of 128 rows on
    // single CTAs halve the resident queries, so the key ring holds two tiles
    // instead of one and the next tile streams in while the current one is
    // used (the second chunk's CTA finds the same keys in L2).  Measured
    // against 256-row chunks on CTA pairs: 0.43 against 0.38-0.42 of HBM.
    const char* pairs = std::getenv("UPF_SCORE_PAIRS");
    const bool pairs_off = pairs && std::strcmp(pairs, "0") == 0;
    const bool pairs_any_d = pairs && std::strcmp(pairs, "1") == 0;
    int qc_max = pl->d <= 128 ? 512 : 256;
    if (pl->d == 256 && pl->QR <= 256) qc_max = 128;
    pl->QC = std::min(((pl->QR + 127) / 128) * 128, qc_max);
    pl->NQC = ceil_div(pl->QR, pl->QC);
    // Tensor-core kernels load tail rows in TMA boxes of 16..128 rows that
    // divide n; other n fall back to the CUDA-core kernels.  UPF_SCORE_PATH=simt
    // forces the CUDA-core kernels (used by tests to cross-check the two).
    pl->q_box_rows = 0;
    for (int rows = 128; rows >= 16; rows >>= 1)
      if (pl->n % rows == 0) {
        pl->q_box_rows = rows;
        break;
      }
    const char* path = std::getenv("UPF_SCORE_PATH");
    pl->use_tc = pl->q_box_rows > 0 && !(path && std::strcmp(path, "simt") == 0);
    // Small batches: when even one key tile per item would leave SMs without
    // an item, smaller query chunks spread the same work over more SMs (every
    // chunk reads its keys again, from L2) and each item runs fewer units in a
    // row.  Halved down to one 128-row tile while the items stay below one
    // per SM.
    if (pl->use_tc) {
      const int tile = upf::score_tc_key_tile(1, pl->d);
      auto most_items = [&](int qc) {
        long long items = 0;
        for (int r = 0; r < pl->R; ++r)
          items += (long long)pl->Hkv * ceil_div(pl->QR, qc) *
                   ceil_div(b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r], tile);
        return items;
      };
      while (pl->QC > 128 && most_items(pl->QC) < upf::kPlanSMs) pl->QC = ((pl->QC / 2 + 127) / 128) * 128;
      pl->NQC = ceil_div(pl->QR, pl->QC);
    }
    // Key splits: the tensor-core kernels hold one CTA per SM, so one wave of
    // about one item per SM; the CUDA-core kernels want a few waves.  The split
    // depends only on the batch and parameters (never on the device), so
    // upf_workspace_bytes() without a context sizes exactly what a call uses.
    (void)ctx;
    // At d = 256, chunks of whole 256-row units run on CTA pairs (one M = 256
    // MMA over two SMs): each SM holds half of the 128 KB query chunk and
    // reads 8 instead of 12 KB of operands per 128 MMA clocks, which the
    // d = 256 passes (MMA-bound, two 64 KB key tiles) need; measured 21-26 %
    // faster there.  At d <= 128 the exponentials match the MMA rate and the
    // pair, whose MMA waits for both CTAs' epilogues, was measured 45 %
    // slower, so those stay on single CTAs.  UPF_SCORE_PAIRS=0 keeps every
    // chunk on single CTAs, =1 allows pairs at any d (tests cross-check both).
    pl->use_pair = pl->use_tc && pl->QC % 256 == 0 && !pairs_off && (pl->d == 256 || pairs_any_d);
    pl->QC2 = pl->QC;
    pl->NQC2 = pl->NQC;
    pl->use_pair2 = pl->use_pair;
    // A d = 256 group of 129..256 rows in a long pass: pass 1 on single CTAs
    // in 128-row chunks (above), pass 2 on CTA pairs in one 256-row chunk that
    // merges both pass-1 chunks' partials.  Measured per pass against one
    // layout for both (Gemma-3 n = 128, 8 kv heads x 128K keys): pass 1 126.5
    // us single against 139 on pairs, pass 2 134 on pairs against 141.4
    // single, step 280 -> 273 us.  With 2 kv heads (Qwen3-Next n = 32) pass 2
    // gained 0.8 us and the step lost 1.6, so shorter passes keep one layout.
    if (pl->use_tc && pl->d == 256 && !pairs_off && pl->QC == 128 && pl->QR > 128 && pl->QR <= 256 &&
        (long long)pl->Hkv * pl->T >= (1LL << 19)) {
      pl->QC2 = 256;
      pl->NQC2 = 1;
      pl->use_pair2 = true;
    }
    if (pl->use_tc) {
      pl->KS1 = pl->use_pair ? choose_split_tc(b, pl->Hkv, pl->NQC, upf::kPairTileKeys, upf::kPlanSMs / 2)
                             : choose_split_tc(b, pl->Hkv, pl->NQC, upf::score_tc_key_tile(1, pl->d), upf::kPlanSMs);
      pl->KS2 = pl->use_pair2 ? choose_split_tc(b, pl->Hkv, pl->NQC2, upf::kPairTileKeys, upf::kPlanSMs / 2)
                              : choose_split_tc(b, pl->Hkv, pl->NQC2, upf::score_tc_key_tile(2, pl->d), upf::kPlanSMs);
    } else {
      pl->KS1 = choose_split(b, pl->Hkv * pl->NQC, 4LL * upf::kPlanSMs, 128);
      pl->KS2 = choose_split(b, pl->Hkv * pl->NQC, 4LL * upf::kPlanSMs, 128);
    }
    pl->pw = pl->use_tc ? upf::kTcPartials : 1;
    pl->items1 = pl->items2 = 0;
    pl->NB = 0;
    pl->max_nb = 0;
    for (int r = 0; r < pl->R; ++r) {
      int L = b->cu_seqlens_host[r + 1] - b->cu_seqlens_host[r];
      pl->items1 += (long long)pl->Hkv * pl->NQC * ceil_div(L, pl->KS1);
      pl->items2 += (long long)pl->Hkv * pl->NQC2 * ceil_div(L, pl->KS2);
      int nb = ceil_div(L, pl->G);
      pl->NB += nb;
      pl->max_nb = std::max(pl->max_nb, nb);
    }
    if (pl->max_nb > upf::kMaxBlocksPerReq)
      return fail(UPF_ERR_UNSUPPORTED, "a request has %d blocks; at most %d are supported", pl->max_nb,
                  upf::kMaxBlocksPerReq);
    if (pl->items1 > (1LL << 30) || pl->items2 > (1LL << 30)) return fail(UPF_ERR_UNSUPPORTED, "batch too large");
    pl->qhead.assign(pl->Hq, 0);
    std::vector<int> fill(pl->Hkv, 0);
    for (int h = 0; h < pl->Hq; ++h) {
      int g = b->kv_of_q ? b->kv_of_q[h] : h / pl->gamma;
      pl->qhead[g * pl->gamma + fill[g]++] = h;
    }
  }
  pl->nwords = ceil_div(pl->T, 32);
  pl->nchunks = std::max(1, ceil_div(pl->nwords, upf::kCompactChunkWords));
  size_t off = 0;
  pl->off_desc = off;
  off = align256(off + sizeof(int32_t) * 3 * (pl->R + 1));
  pl->off_p1 = off;
  off = align256(off + sizeof(float2) * size_t(pl->items1) * pl->pw * pl->QC);
  pl->off_part = off;
  off = align256(off + sizeof(float) * size_t(pl->Hkv) * pl->NQC2 * pl->pw * pl->T);
  pl->off_bs = off;
  off = align256(off + sizeof(float) * size_t(pl->NB));
  pl->off_chunk = off;
  off = align256(off + sizeof(int32_t) * pl->nchunks);
  pl->off_kidx = off;
  off = align256(off + sizeof(int32_t) * size_t(pl->T));
  pl->off_ctr = off;   // tail counters [R+1], then edge words [2R]
  off = align256(off + sizeof(int32_t) * size_t(pl->R + 1) + sizeof(uint32_t) * 2 * size_t(pl->R));
  pl->off_kbl = off;   // kept blocks [NB], their output offsets [NB], kept blocks per request [R]
  off = align256(off + sizeof(int32_t) * (2 * size_t(pl->NB) + size_t(pl->R)));
  pl->total = off;
  pl->nonempty = 0;
  for (int r = 0; r < pl->R; ++r) pl->nonempty += b->cu_seqlens_host[r + 1] > b->cu_seqlens_host[r];
  return UPF_OK;
}

upf_status check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (!ws) return fail(UPF_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(UPF_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < pl.total)
    return fail(UPF_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, pl.total);
  return UPF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

upf_status check_ctx(const upf_ctx* ctx) {
  if (!ctx) return fail(UPF_ERR_INVALID_ARG, "context is NULL");
  return UPF_OK;
}

upf_status check_score_io(const Plan& pl, const void* q, int64_t qs, const void* k, int64_t ks) {
  if (!q || !k) return fail(UPF_ERR_INVALID_ARG, "q and k are required");
  if (!aligned16(q) || !aligned16(k)) return fail(UPF_ERR_INVALID_ARG, "q and k must be 16-byte aligned");
  if (qs < (int64_t)pl.Hq * pl.d || qs % 8) return fail(UPF_ERR_INVALID_ARG, "q_row_stride must be >= H_q*d and a multiple of 8");
  if (ks < (int64_t)pl.Hkv * pl.d || ks % 8) return fail(UPF_ERR_INVALID_ARG, "k_row_stride must be >= H_kv*d and a multiple of 8");
  return UPF_OK;
}

// A compaction buffer the kernels may dereference: device or managed memory,
// page-locked host memory mapped at the same address (unified addressing), or
// any host memory when the device reads pageable memory itself.
bool device_accessible(const void* p, int device) {
  if (!p) return true;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return true;
    case cudaMemoryTypeHost:
      return at.devicePointer == p;
    default: {
      int pageable = 0;
      return cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, device) == cudaSuccess && pageable;
    }
  }
}

upf_status check_compact_io(const Plan& pl, const uint32_t* keep_bits, const upf_compact_io* io, int device) {
  if (!keep_bits) return fail(UPF_ERR_INVALID_ARG, "keep_bits is NULL");
  if (!io) return fail(UPF_ERR_INVALID_ARG, "compact io is NULL");
  if (!io->cu_seqlens_out || !io->total_kept) return fail(UPF_ERR_INVALID_ARG, "cu_seqlens_out and total_kept are required");
  if (!io->hidden_in != !io->hidden_out) return fail(UPF_ERR_INVALID_ARG, "hidden_in/hidden_out must both be set or both NULL");
  if (!io->pos_in != !io->pos_out) return fail(UPF_ERR_INVALID_ARG, "pos_in/pos_out must both be set or both NULL");
  if (!io->slot_in != !io->slot_out) return fail(UPF_ERR_INVALID_ARG, "slot_in/slot_out must both be set or both NULL");
  if (io->hidden_in) {
    if (io->row_bytes <= 0 || io->row_bytes % 16) return fail(UPF_ERR_INVALID_ARG, "row_bytes must be a positive multiple of 16");
    if (!aligned16(io->hidden_in) || !aligned16(io->hidden_out))
      return fail(UPF_ERR_INVALID_ARG, "hidden buffers must be 16-byte aligned");
  }
  const void* bufs[6] = {io->hidden_in, io->hidden_out, io->pos_in, io->pos_out, io->slot_in, io->slot_out};
  static const char* names[6] = {"hidden_in", "hidden_out", "pos_in", "pos_out", "slot_in", "slot_out"};
  for (int i = 0; i < 6; ++i)
    if (!device_accessible(bufs[i], device))
      return fail(UPF_ERR_INVALID_ARG, "%s is host memory the device cannot access (use page-locked memory)", names[i]);
  if (!io->history != !io->history_len) return fail(UPF_ERR_INVALID_ARG, "history/history_len must both be set or both NULL");
  if (io->history && io->history_cap < 1) return fail(UPF_ERR_INVALID_ARG, "history_cap must be >= 1");
  (void)pl;
  return UPF_OK;
}

upf::ScoreArgs score_args(const upf_ctx* ctx, const upf_batch* b, const Plan& pl, const void* q, int64_t qs,
                          const void* k, int64_t ks, void* ws) {
  upf::ScoreArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.q_stride = qs;
  a.k_stride = ks;
  a.cu = b->cu_seqlens_dev;
  a.R = pl.R;
  a.T = pl.T;
  a.Hq = pl.Hq;
  a.Hkv = pl.Hkv;
  a.d = pl.d;
  a.n = pl.n;
  a.gamma = pl.gamma;
  a.QR = pl.QR;
  a.QC = pl.QC;     // pass 1's chunks; pass2_args() switches to pass 2's
  a.NQC = pl.NQC;
  a.QC1 = pl.QC;
  a.NQC1 = pl.NQC;
  a.KS1 = pl.KS1;
  a.KS2 = pl.KS2;
  a.items1 = int(pl.items1);
  a.items2 = int(pl.items2);
  a.scale_log2 = pl.scale * 1.4426950408889634f;
  a.q_box_rows = pl.q_box_rows;
  a.use_tc = pl.use_tc ? 1 : 0;
  a.use_pair = pl.use_pair ? 1 : 0;
  a.item_off1 = at<int32_t>(ws, pl.off_desc);
  a.item_off2 = at<int32_t>(ws, pl.off_desc) + (pl.R + 1);
  a.pw = pl.pw;
  a.p1part = at<float2>(ws, pl.off_p1);
  a.part = at<float>(ws, pl.off_part);
  a.status = ctx->status_dev;
  a.wait_limit = ctx->wait_limit > 0 ? ctx->wait_limit : upf::kDefaultWaitCycles;
  for (int i = 0; i < pl.Hq; ++i) a.qhead[i] = pl.qhead[i];
  return a;
}

// Pass 2's arguments: pass 1's with pass 2's query chunks and kernel kind
// (QC1 / NQC1 keep pass 1's, where the pass-1 partials are).
upf::ScoreArgs pass2_args(const upf::ScoreArgs& a1, const Plan& pl) {
  upf::ScoreArgs a = a1;
  a.QC = pl.QC2;
  a.NQC = pl.NQC2;
  a.use_pair = pl.use_pair2 ? 1 : 0;
  return a;
}

upf::DescribeArgs describe_args(const upf_ctx* ctx, const upf_batch* b, const Plan& pl, void* ws) {
  upf::DescribeArgs a;
  a.cu = b->cu_seqlens_dev;
  a.R = pl.R;
  a.T = pl.T;
  a.Hkv = pl.Hkv;
  a.NQC = pl.NQC;
  a.NQC2 = pl.NQC2;
  a.KS1 = pl.KS1;
  a.KS2 = pl.KS2;
  a.G = pl.G;
  a.items1 = int(pl.items1);
  a.items2 = int(pl.items2);
  a.NB = int(pl.NB);
  a.item_off1 = at<int32_t>(ws, pl.off_desc);
  a.item_off2 = a.item_off1 + (pl.R + 1);
  a.blk_off = a.item_off2 + (pl.R + 1);
  a.status = ctx->status_dev;
  a.counters = at<int32_t>(ws, pl.off_ctr);
  a.ncounters = pl.R + 1;
  return a;
}

// The tables describe_kernel would build, from cu_seqlens_host (the batch has
// at most kInlineReqs requests).
void fill_desc(const upf_batch* b, const Plan& pl, upf::DescInline* d) {
  const int32_t* cu = b->cu_seqlens_host;
  const int units1 = pl.Hkv * pl.NQC, units2 = pl.Hkv * pl.NQC2;
  int o1 = 0, o2 = 0, ob = 0;
  d->R = pl.R;
  for (int r = 0; r <= pl.R; ++r) {
    d->cu[r] = cu[r];
    d->off1[r] = o1;
    d->off2[r] = o2;
    d->blk[r] = ob;
    if (r == pl.R) break;
    const int L = cu[r + 1] - cu[r];
    o1 += units1 * ceil_div(L, pl.KS1);
    o2 += units2 * ceil_div(L, pl.KS2);
    ob += ceil_div(L, pl.G);
  }
}

// Arguments of the fused tail; with_lists: the kept-block lists for the
// gather; cu_out / total_kept nullable.
upf::TailArgs tail_args(const upf::SelectArgs& se, const Plan& pl, void* ws, bool with_lists, int32_t* cu_out,
                        int32_t* total_kept) {
  upf::TailArgs t;
  t.s = se;
  t.counters = at<int32_t>(ws, pl.off_ctr);
  t.edge_bits = reinterpret_cast<uint32_t*>(t.counters + (pl.R + 1));
  t.kept_blk = with_lists ? at<int32_t>(ws, pl.off_kbl) : nullptr;
  t.kept_off = with_lists ? t.kept_blk + pl.NB : nullptr;
  t.kept_nblk = with_lists ? t.kept_blk + 2 * pl.NB : nullptr;
  t.cu_out = cu_out;
  t.total_kept = total_kept;
  t.nonempty = pl.nonempty;
  t.bpc = upf::tail_blocks_per_cta(pl.G);
  t.nbp = ((pl.max_nb > 0 ? pl.max_nb : 1) + 7) & ~7;
  t.desc.R = 0;
  return t;
}

upf::SelectArgs select_args(const upf_ctx* ctx, const upf_batch* b, const Plan& pl, void* ws, int P,
                            const float* part, const float* scores_in, float* scores_out, float* block_scores,
                            uint32_t* keep_bits, int32_t* kept_count) {
  upf::SelectArgs a;
  a.cu = b->cu_seqlens_dev;
  a.R = pl.R;
  a.T = pl.T;
  a.G = pl.G;
  a.sink_keep = pl.sink;
  a.tail_keep = pl.tail;
  a.n = pl.n;
  a.Hq = pl.Hq;
  a.NB = int(pl.NB);
  a.max_nb = pl.max_nb;
  a.P = P;
  a.top_p = pl.top_p;
  a.part = part;
  a.scores_in = scores_in;
  a.scores_out = scores_out;
  a.block_scores = block_scores ? block_scores : at<float>(ws, pl.off_bs);
  a.blk_off = at<int32_t>(ws, pl.off_desc) + 2 * (pl.R + 1);
  a.keep_bits = keep_bits;
  a.kept_count = kept_count;
  a.status = ctx->status_dev;
  return a;
}

upf::CompactArgs compact_args(const upf_ctx* ctx, const upf_batch* b, const Plan& pl, const uint32_t* keep_bits,
                              const upf_compact_io* io, void* ws) {
  upf::CompactArgs a;
  a.cu = b->cu_seqlens_dev;
  a.R = pl.R;
  a.T = pl.T;
  a.nwords = pl.nwords;
  a.nchunks = pl.nchunks;
  a.keep_bits = keep_bits;
  a.chunk_tot = at<int32_t>(ws, pl.off_chunk);
  a.kept_index = io->kept_index ? io->kept_index : at<int32_t>(ws, pl.off_kidx);
  a.row_bytes = io->hidden_in ? io->row_bytes : 0;
  a.hidden_in = io->hidden_in;
  a.hidden_out = io->hidden_out;
  a.pos_in = io->pos_in;
  a.pos_out = io->pos_out;
  a.slot_in = io->slot_in;
  a.slot_out = io->slot_out;
  a.cu_out = io->cu_seqlens_out;
  a.total_kept = io->total_kept;
  a.layer_id = io->layer_id;
  a.history_cap = io->history_cap;
  a.history = io->history;
  a.history_len = io->history_len;
  a.status = ctx->status_dev;
  return a;
}

#define UPF_LAUNCH(expr, what)                       \
  do {                                               \
    cudaError_t e_ = (expr);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Launch `f` as stage `stage`: counted always, bracketed by events when tracing.
template <class F>
cudaError_t staged(upf_ctx* ctx, int stage, cudaStream_t s, F&& f) {
  ctx->launches[stage]++;
  if (!ctx->profiling) return f();
  cudaEvent_t a = ctx->event(), b = ctx->event();
  if (!a || !b) return cudaErrorMemoryAllocation;
  cudaEventRecord(a, s);
  cudaError_t e = f();
  cudaEventRecord(b, s);
  ctx->pending.push_back({stage, a, b});
  return e;
}

enum Stage { kDescribe = 0, kPass1, kPass2, kFinalize, kSelect, kCompactCount, kCompactIndex, kCompactGather };

// chained: the first compaction kernel follows another kernel of the same call
// (PDL).  A batch of one chunk needs no chunk totals: its index kernel starts
// from zero.
upf_status launch_compact_all(upf_ctx* ctx, const upf::CompactArgs& ca, cudaStream_t s, bool chained) {
  if (ca.nchunks > 1)
    UPF_LAUNCH(staged(ctx, kCompactCount, s, [&] { return upf::launch_compact_count(ca, s, chained); }),
               "compact count");
  const bool index_chained = ca.nchunks > 1 || chained;
  UPF_LAUNCH(staged(ctx, kCompactIndex, s, [&] { return upf::launch_compact_index(ca, s, index_chained); }),
             "compact index");
  UPF_LAUNCH(staged(ctx, kCompactGather, s, [&] { return upf::launch_compact_gather(ca, s, true); }), "compact gather");
  return UPF_OK;
}

}  // namespace

void upf::set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

extern "C" {

int upf_version(void) { return UPF_VERSION; }

void upf_default_params(upf_params* p) {
  if (!p) return;
  p->n_tail = 128;
  p->block = 64;
  p->sink_keep = 128;
  p->tail_keep = 128;
  p->top_p = 0.99f;
  p->softmax_scale = 0.f;
}

const char* upf_status_name(upf_status s) {
  switch (s) {
    case UPF_OK: return "UPF_OK";
    case UPF_ERR_INVALID_ARG: return "UPF_ERR_INVALID_ARG";
    case UPF_ERR_UNSUPPORTED: return "UPF_ERR_UNSUPPORTED";
    case UPF_ERR_CUDA: return "UPF_ERR_CUDA";
    case UPF_ERR_CAPACITY: return "UPF_ERR_CAPACITY";
    case UPF_ERR_NONFINITE: return "UPF_ERR_NONFINITE";
    case UPF_ERR_TIMEOUT: return "UPF_ERR_TIMEOUT";
  }
  return "UPF_ERR_UNKNOWN";
}

const char* upf_last_error(void) { return g_last_error.c_str(); }

upf_status upf_create(upf_ctx** out, int device) {
  if (!out) return fail(UPF_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= count) return fail(UPF_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, count);
  DeviceGuard guard(device);
  if (!guard.ok) return fail(UPF_ERR_CUDA, "cudaSetDevice(%d) failed", device);
  upf_ctx* c = new upf_ctx();
  c->device = device;
  if ((e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  if (major * 10 + minor != 103) {
    delete c;
    return fail(UPF_ERR_UNSUPPORTED, "libupf is built for sm_103a; device %d is sm_%d%d", device, major, minor);
  }
  if ((e = cudaMalloc(&c->status_dev, 64 * sizeof(int32_t))) != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaMalloc(status)");
  }
  if ((e = cudaMemset(c->status_dev, 0, 64 * sizeof(int32_t))) != cudaSuccess) {
    cudaFree(c->status_dev);
    delete c;
    return cuda_fail(e, "cudaMemset(status)");
  }
  *out = c;
  return UPF_OK;
}

upf_status upf_destroy(upf_ctx* ctx) {
  if (!ctx) return fail(UPF_ERR_INVALID_ARG, "context is NULL");
  DeviceGuard guard(ctx->device);
  for (auto& r : ctx->pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : ctx->pool) cudaEventDestroy(e);
  cudaFree(ctx->status_dev);
  delete ctx;
  return UPF_OK;
}

upf_status upf_sync_status(upf_ctx* ctx, void* stream) {
  upf_status st = check_ctx(ctx);
  if (st != UPF_OK) return st;
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t code = 0;
  if ((e = cudaMemcpy(&code, ctx->status_dev, sizeof(code), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status");
  if (code != 0) {
    if ((e = cudaMemset(ctx->status_dev, 0, sizeof(int32_t))) != cudaSuccess) return cuda_fail(e, "reset status");
    return fail(static_cast<upf_status>(code), "device reported %s", upf_status_name(static_cast<upf_status>(code)));
  }
  return UPF_OK;
}

const char* upf_stage_name(int32_t stage) {
  static const char* names[UPF_NUM_STAGES] = {"describe",       "score_pass1",   "score_pass2",  "finalize",
                                              "select",         "compact_count", "compact_index", "compact_gather"};
  return (stage >= 0 && stage < UPF_NUM_STAGES) ? names[stage] : "";
}

upf_status upf_profile_enable(upf_ctx* ctx, int32_t on) {
  upf_status st = check_ctx(ctx);
  if (st != UPF_OK) return st;
  ctx->profiling = on != 0;
  return UPF_OK;
}

upf_status upf_profile_read(upf_ctx* ctx, int32_t* launches, double* ms, int32_t n_stages) {
  upf_status st = check_ctx(ctx);
  if (st != UPF_OK) return st;
  if (n_stages < 0 || n_stages > UPF_NUM_STAGES) return fail(UPF_ERR_INVALID_ARG, "n_stages must be in [0, %d]", UPF_NUM_STAGES);
  DeviceGuard guard(ctx->device);
  double acc[UPF_NUM_STAGES] = {};
  cudaError_t err = cudaSuccess;
  for (auto& r : ctx->pending) {
    cudaError_t e = cudaEventSynchronize(r.b);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
    if (e != cudaSuccess && err == cudaSuccess) err = e;
    acc[r.stage] += t;
    ctx->pool.push_back(r.a);
    ctx->pool.push_back(r.b);
  }
  ctx->pending.clear();
  for (int i = 0; i < n_stages; ++i) {
    if (launches) launches[i] = ctx->launches[i];
    if (ms) ms[i] = acc[i];
  }
  for (int i = 0; i < UPF_NUM_STAGES; ++i) ctx->launches[i] = 0;
  if (err != cudaSuccess) return cuda_fail(err, "profile events");
  return UPF_OK;
}

size_t upf_workspace_bytes(const upf_batch* batch, const upf_params* params) {
  Plan pl;
  if (make_plan(nullptr, batch, params, true, &pl) != UPF_OK) return 0;
  return pl.total;
}

// upf_score and upf_score_shard: scores normalised by hq_norm q heads (the
// batch's own H_q, or the total over tensor-parallel ranks).
static upf_status score_impl(upf_ctx* ctx, const upf_batch* batch, const upf_params* params, int hq_norm,
                             const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                             float* scores, void* ws, size_t ws_bytes, void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  Plan pl;
  if ((st = make_plan(ctx, batch, params, true, &pl)) != UPF_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != UPF_OK) return st;
  if ((st = check_score_io(pl, q, q_row_stride, k, k_row_stride)) != UPF_OK) return st;
  if (!scores) return fail(UPF_ERR_INVALID_ARG, "scores is NULL");
  if (hq_norm < pl.Hq || hq_norm > (1 << 20))
    return fail(UPF_ERR_INVALID_ARG, "num_q_heads_total (%d) must be in [num_q_heads (%d), 2^20]", hq_norm, pl.Hq);
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const upf::DescribeArgs da = describe_args(ctx, batch, pl, ws);
  UPF_LAUNCH(staged(ctx, kDescribe, s, [&] { return upf::launch_describe(da, s, false); }), "describe");
  upf::ScoreArgs sa = score_args(ctx, batch, pl, q, q_row_stride, k, k_row_stride, ws);
  UPF_LAUNCH(staged(ctx, kPass1, s, [&] { return upf::launch_score_pass1(sa, s, true); }), "score pass 1");
  UPF_LAUNCH(staged(ctx, kPass2, s, [&] { return upf::launch_score_pass2(pass2_args(sa, pl), s, true); }), "score pass 2");
  upf::SelectArgs se = select_args(ctx, batch, pl, ws, pl.Hkv * pl.NQC2 * pl.pw, sa.part, nullptr, scores, nullptr,
                                   nullptr, nullptr);
  se.Hq = hq_norm;
  UPF_LAUNCH(staged(ctx, kFinalize, s, [&] { return upf::launch_block_means(se, s, true); }), "finalize scores");
  return UPF_OK;
}

upf_status upf_plan_info(const upf_batch* batch, const upf_params* params, int32_t* key_split1, int32_t* key_split2,
                         int64_t* items1, int64_t* items2, int32_t* ctas_per_item1, int32_t* ctas_per_item2) {
  Plan pl;
  upf_status st = make_plan(nullptr, batch, params, true, &pl);
  if (st != UPF_OK) return st;
  if (key_split1) *key_split1 = pl.KS1;
  if (key_split2) *key_split2 = pl.KS2;
  if (items1) *items1 = pl.items1;
  if (items2) *items2 = pl.items2;
  if (ctas_per_item1) *ctas_per_item1 = pl.use_pair ? 2 : 1;
  if (ctas_per_item2) *ctas_per_item2 = pl.use_pair2 ? 2 : 1;
  return UPF_OK;
}

upf_status upf_score(upf_ctx* ctx, const upf_batch* batch, const upf_params* params, const void* q,
                     int64_t q_row_stride, const void* k, int64_t k_row_stride, float* scores, void* ws,
                     size_t ws_bytes, void* stream) {
  if (!batch) return fail(UPF_ERR_INVALID_ARG, "batch is NULL");
  return score_impl(ctx, batch, params, batch->num_q_heads, q, q_row_stride, k, k_row_stride, scores, ws, ws_bytes,
                    stream);
}

upf_status upf_score_shard(upf_ctx* ctx, const upf_batch* batch, const upf_params* params,
                           int32_t num_q_heads_total, const void* q, int64_t q_row_stride, const void* k,
                           int64_t k_row_stride, float* scores, void* ws, size_t ws_bytes, void* stream) {
  return score_impl(ctx, batch, params, num_q_heads_total, q, q_row_stride, k, k_row_stride, scores, ws, ws_bytes,
                    stream);
}

upf_status upf_set_wait_limit(upf_ctx* ctx, int64_t cycles) {
  upf_status st = check_ctx(ctx);
  if (st != UPF_OK) return st;
  if (cycles < 0) return fail(UPF_ERR_INVALID_ARG, "wait limit must be >= 0 cycles (0 restores the default)");
  ctx->wait_limit = cycles;
  return UPF_OK;
}

upf_status upf_select(upf_ctx* ctx, const upf_batch* batch, const upf_params* params, const float* scores,
                      float* block_scores, uint32_t* keep_bits, int32_t* kept_count, void* ws, size_t ws_bytes,
                      void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  Plan pl;
  if ((st = make_plan(ctx, batch, params, true, &pl)) != UPF_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != UPF_OK) return st;
  if (!scores || !keep_bits || !kept_count) return fail(UPF_ERR_INVALID_ARG, "scores, keep_bits and kept_count are required");
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const upf::DescribeArgs da = describe_args(ctx, batch, pl, ws);
  UPF_LAUNCH(staged(ctx, kDescribe, s, [&] { return upf::launch_describe(da, s, false); }), "describe");
  upf::SelectArgs se = select_args(ctx, batch, pl, ws, 0, nullptr, scores, nullptr, block_scores, keep_bits,
                                   kept_count);
  if (fused_tail(pl)) {
    const upf::TailArgs ta = tail_args(se, pl, ws, false, nullptr, nullptr);
    UPF_LAUNCH(staged(ctx, kSelect, s, [&] { return upf::launch_tail(ta, s, true); }), "block means and select");
    return UPF_OK;
  }
  UPF_LAUNCH(staged(ctx, kFinalize, s, [&] { return upf::launch_block_means(se, s, true); }), "block means");
  UPF_LAUNCH(staged(ctx, kSelect, s, [&] { return upf::launch_select(se, s, true); }), "select");
  return UPF_OK;
}

upf_status upf_compact(upf_ctx* ctx, const upf_batch* batch, const uint32_t* keep_bits, const upf_compact_io* io,
                       void* ws, size_t ws_bytes, void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  Plan pl;
  if ((st = make_plan(ctx, batch, nullptr, false, &pl)) != UPF_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != UPF_OK) return st;
  if ((st = check_compact_io(pl, keep_bits, io, ctx->device)) != UPF_OK) return st;
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_compact_all(ctx, compact_args(ctx, batch, pl, keep_bits, io, ws), s, false);
}

upf_status upf_revive(upf_ctx* ctx, const upf_batch* batch, const int32_t* kept_index, const int32_t* total_kept,
                      const void* rows, int64_t row_bytes, void* full, void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  if ((st = check_batch(batch)) != UPF_OK) return st;
  if (!kept_index || !total_kept || !rows || !full) return fail(UPF_ERR_INVALID_ARG, "kept_index, total_kept, rows and full are required");
  if (row_bytes <= 0 || row_bytes % 16) return fail(UPF_ERR_INVALID_ARG, "row_bytes must be a positive multiple of 16");
  if (!aligned16(rows) || !aligned16(full)) return fail(UPF_ERR_INVALID_ARG, "rows and full must be 16-byte aligned");
  DeviceGuard guard(ctx->device);
  upf::ReviveArgs a;
  a.T = batch->cu_seqlens_host[batch->num_reqs];
  a.kept_index = kept_index;
  a.total_kept = total_kept;
  a.rows = rows;
  a.full = full;
  a.row_bytes = row_bytes;
  UPF_LAUNCH(upf::launch_revive(a, static_cast<cudaStream_t>(stream)), "revive");
  return UPF_OK;
}

upf_status upf_history_kv_len(upf_ctx* ctx, const upf_batch* batch, const int32_t* history,
                              const int32_t* history_len, int32_t history_cap, int32_t layer_id, int32_t* kv_len,
                              void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  if ((st = check_batch(batch)) != UPF_OK) return st;
  if (!history || !history_len || !kv_len) return fail(UPF_ERR_INVALID_ARG, "history, history_len and kv_len are required");
  if (history_cap < 1) return fail(UPF_ERR_INVALID_ARG, "history_cap must be >= 1");
  DeviceGuard guard(ctx->device);
  upf::HistoryArgs a;
  a.cu = batch->cu_seqlens_dev;
  a.R = batch->num_reqs;
  a.layer_id = layer_id;
  a.history_cap = history_cap;
  a.history = history;
  a.history_len = history_len;
  a.kv_len = kv_len;
  UPF_LAUNCH(upf::launch_history_kv_len(a, static_cast<cudaStream_t>(stream)), "history kv length");
  return UPF_OK;
}

upf_status upf_select_tokens(upf_ctx* ctx, const upf_batch* batch, const upf_params* params, const void* q,
                             int64_t q_row_stride, const void* k, int64_t k_row_stride, float* scores,
                             float* block_scores, uint32_t* keep_bits, int32_t* kept_count,
                             const upf_compact_io* io, void* ws, size_t ws_bytes, void* stream) {
  upf_status st;
  if ((st = check_ctx(ctx)) != UPF_OK) return st;
  Plan pl;
  if ((st = make_plan(ctx, batch, params, true, &pl)) != UPF_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != UPF_OK) return st;
  if ((st = check_score_io(pl, q, q_row_stride, k, k_row_stride)) != UPF_OK) return st;
  if (!keep_bits || !kept_count) return fail(UPF_ERR_INVALID_ARG, "keep_bits and kept_count are required");
  if ((st = check_compact_io(pl, keep_bits, io, ctx->device)) != UPF_OK) return st;
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  upf::ScoreArgs sa = score_args(ctx, batch, pl, q, q_row_stride, k, k_row_stride, ws);
  // Batches of up to kInlineReqs requests on the tensor-core path carry the
  // descriptor tables in the kernel parameters: no describe launch, and pass 1
  // checks the device cu_seqlens and clears the tail's counters instead.
  const bool carried = pl.use_tc && fused_tail(pl) && pl.R <= upf::kInlineReqs && pl.items1 > 0 && pl.items2 > 0;
  if (carried) {
    fill_desc(batch, pl, &sa.desc);
    sa.counters = at<int32_t>(ws, pl.off_ctr);
    sa.ncounters = pl.R + 1;
  } else {
    const upf::DescribeArgs da = describe_args(ctx, batch, pl, ws);
    UPF_LAUNCH(staged(ctx, kDescribe, s, [&] { return upf::launch_describe(da, s, false); }), "describe");
  }
  UPF_LAUNCH(staged(ctx, kPass1, s, [&] { return upf::launch_score_pass1(sa, s, true); }), "score pass 1");
  UPF_LAUNCH(staged(ctx, kPass2, s, [&] { return upf::launch_score_pass2(pass2_args(sa, pl), s, true); }), "score pass 2");
  upf::SelectArgs se = select_args(ctx, batch, pl, ws, pl.Hkv * pl.NQC2 * pl.pw, sa.part, nullptr, scores, block_scores,
                                   keep_bits, kept_count);
  if (fused_tail(pl)) {
    // finalize + block means + select + kept-block lists + compacted offsets
    // in one launch, then the gather driven by the kept-block lists
    upf::TailArgs ta = tail_args(se, pl, ws, true, io->cu_seqlens_out, io->total_kept);
    if (carried) ta.desc = sa.desc;
    UPF_LAUNCH(staged(ctx, kSelect, s, [&] { return upf::launch_tail(ta, s, true); }), "finalize and select");
    upf::GatherListArgs ga;
    ga.c = compact_args(ctx, batch, pl, keep_bits, io, ws);
    ga.c.kept_index = io->kept_index;   // nullable: written only if the caller asks
    ga.blk_off = se.blk_off;
    ga.kept_blk = ta.kept_blk;
    ga.kept_off = ta.kept_off;
    ga.kept_nblk = ta.kept_nblk;
    ga.G = pl.G;
    ga.desc.R = 0;
    if (carried) ga.desc = sa.desc;
    UPF_LAUNCH(staged(ctx, kCompactGather, s, [&] { return upf::launch_gather_list(ga, s, true); }), "compact gather");
    return UPF_OK;
  }
  UPF_LAUNCH(staged(ctx, kFinalize, s, [&] { return upf::launch_block_means(se, s, true); }), "finalize scores");
  UPF_LAUNCH(staged(ctx, kSelect, s, [&] { return upf::launch_select(se, s, true); }), "select");
  return launch_compact_all(ctx, compact_args(ctx, batch, pl, keep_bits, io, ws), s, true);
}

}  // extern "C"
