// The tail of the per-layer path after scoring: finalize, block means,
// top-p selection with exemption, the keep mask and the kept-token list, in
// one launch; then the gather of the kept rows.
//
// UniPrefill article, section 二 second step (average the token scores inside
// each block of G tokens, keep the smallest block set reaching p of the total
// importance), the exemption paragraph (the first and last 128 tokens are
// always kept), section 二 third step and section 三 (later layers see only
// the kept tokens; positions, slot ids and the batch offsets follow the drop;
// the decision stays on the GPU).
//
// tail_kernel: CTA c owns a run of consecutive blocks of the packed batch
// (bpc blocks; a run may cross request boundaries).  Phase 1, every CTA: each
// token's score (the sum of its per-group partials times 1/(H_q n_eff), or
// the given score) and each block's mean.  Then each CTA counts itself done on
// every request its run touches (one atomic per request); the CTA that
// completes a request runs that request's selection (select_core.cuh) with all
// its threads, writes the request's keep bits, its kept count and the list of
// its kept blocks with their output offsets, and counts the request done.  The
// CTA that completes the last request writes the compacted batch offsets, the
// total, the keep-bit words shared by neighbouring requests, and zero counts
// for empty requests (a batch of one request needs none of that: its
// selecting CTA writes every word and the offsets itself).  Nothing waits:
// completion is detected with fenced atomics, so there is no spin anywhere.
//
// The per-token and per-block sums follow the same order as the separate
// finalize kernel (partials in index order, then tokens lane-strided within a
// warp and a fixed shuffle tree), so the fused and the separate entry points
// give the same bits.
#include <climits>

#include "select_core.cuh"
#include "upf_internal.cuh"

namespace upf {

namespace {

constexpr int kTailThreads = kSelThreads;   // 1024
constexpr int kTailWarps = kTailThreads / 32;

// Counter increment with acquire-release semantics at GPU scope: it publishes
// what this CTA wrote before the preceding barrier and, when it returns the
// final count, makes the other CTAs' published writes visible to this CTA
// (after the next barrier).
__device__ __forceinline__ int add_acq_rel(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ int owner_of(const int32_t* off, int R, int x) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// cu_seqlens and block offsets of a tail or gather launch: those carried in its
// parameters (the argument must be the kernel's __grid_constant__ parameter),
// else the device cu_seqlens and the workspace offsets describe_kernel wrote.
__device__ __forceinline__ DescView tail_view(const TailArgs& a) {
  if (a.desc.R > 0) return DescView{a.desc.cu, nullptr, nullptr, a.desc.blk};
  return DescView{a.s.cu, nullptr, nullptr, a.s.blk_off};
}

__device__ __forceinline__ DescView gather_view(const GatherListArgs& g) {
  if (g.desc.R > 0) return DescView{g.desc.cu, nullptr, nullptr, g.desc.blk};
  return DescView{g.c.cu, nullptr, nullptr, g.blk_off};
}

// The last request is done: offsets of the compacted batch, the total, the
// keep-bit words shared by neighbouring requests (cleared, then the edge bits
// of every request OR-ed in), and zero counts for empty requests.  Run by
// the whole CTA.  With no blocks at all (an empty batch, or a descriptor the
// describe kernel rejected), every count is 0 and every keep bit is cleared.
__device__ void finish_batch(const TailArgs& a, const DescView& dv, bool no_blocks) {
  __shared__ int s_carry;
  __shared__ int s_warp[kTailWarps];
  const SelectArgs& s = a.s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (no_blocks) {
    const int nwords = (s.T + 31) / 32;
    for (int w = tid; w < nwords; w += blockDim.x) s.keep_bits[w] = 0u;
    for (int r = tid; r < s.R; r += blockDim.x) s.kept_count[r] = 0;
  } else {
    for (int r = tid; r < s.R; r += blockDim.x)
      if (dv.cu[r + 1] == dv.cu[r]) s.kept_count[r] = 0;
    // words a request covers only in part: clear, then OR in every request's part
    for (int r = tid; r < s.R; r += blockDim.x) {
      const int tok0 = dv.cu[r], L = dv.cu[r + 1] - tok0;
      if (L <= 0) continue;
      const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
      if (w0 * 32 < tok0 || w0 * 32 + 32 > tok0 + L) s.keep_bits[w0] = 0u;
      if (w1 != w0 && w1 * 32 + 32 > tok0 + L) s.keep_bits[w1] = 0u;
    }
    __syncthreads();
    for (int r = tid; r < s.R; r += blockDim.x) {
      const int tok0 = dv.cu[r], L = dv.cu[r + 1] - tok0;
      if (L <= 0) continue;
      const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
      if (w0 * 32 < tok0 || w0 * 32 + 32 > tok0 + L) atomicOr(&s.keep_bits[w0], __ldcg(a.edge_bits + 2 * r));
      if (w1 != w0 && w1 * 32 + 32 > tok0 + L) atomicOr(&s.keep_bits[w1], __ldcg(a.edge_bits + 2 * r + 1));
    }
  }
  if (!a.cu_out) return;
  // cu_out = exclusive prefix of the kept counts, in chunks of blockDim.x requests
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < s.R; base += blockDim.x) {
    const int r = base + tid;
    const int v = (r < s.R && !no_blocks) ? __ldcg(s.kept_count + r) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    const int before = s_carry + warps_before_sum(s_warp);
    if (r < s.R) a.cu_out[r] = before + incl - v;
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry = before + incl;
    __syncthreads();
  }
  if (tid == 0) {
    a.cu_out[s.R] = s_carry;
    *a.total_kept = s_carry;
  }
}

// Selection of request r by the whole CTA, then its keep bits (whole words
// inside the request by plain stores, the first and last word's bits to the
// edge scratch unless the batch is this one request), its count and its
// kept-token list.  Returns the kept-token count.
__device__ int select_and_emit(const TailArgs& a, const DescView& dv, int r, const SelectScratch& sc) {
  __shared__ int s_warpb[kTailWarps];
  const SelectArgs& s = a.s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = dv.blk[r], nb = dv.blk[r + 1] - b0;
  const int tok0 = dv.cu[r], L = dv.cu[r + 1] - tok0;
  const int kept = select_request(s.block_scores + b0, nb, L, s.G, s.top_p, s.sink_keep, s.tail_keep, sc, s.status);
  const int w0 = tok0 >> 5, w1 = (tok0 + L - 1) >> 5;
  const int gshift = block_shift(s.G);
  for (int w = w0 + tid; w <= w1; w += blockDim.x) {
    const uint32_t bits = request_word_bits(sc.keep, tok0, L, s.G, gshift, w);
    const bool partial = s.R > 1 && ((w * 32 < tok0) || (w * 32 + 32 > tok0 + L));
    if (!partial) {
      s.keep_bits[w] = bits;
    } else {   // read by the CTA that finishes the batch
      a.edge_bits[2 * r + (w == w0 ? 0 : 1)] = bits;
    }
  }
  if (a.kept_blk) {
    // The kept blocks in order with their output offsets inside the request
    // (every block but the request's last holds G tokens, so a kept block's
    // offset is G times the number of kept blocks before it); thread t owns
    // the contiguous blocks [t*per, (t+1)*per).  The gather expands them to
    // token rows.
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int i0 = min(nb, tid * per), i1 = min(nb, i0 + per);
    int mineb = 0;
    for (int i = i0; i < i1; ++i) mineb += sc.keep[i] ? 1 : 0;
    int inclb = mineb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tb = __shfl_up_sync(0xffffffffu, inclb, o);
      if (lane >= o) inclb += tb;
    }
    if (lane == 31) s_warpb[warp] = inclb;
    __syncthreads();
    int runb = inclb - mineb + warps_before_sum(s_warpb);
    for (int i = i0; i < i1; ++i)
      if (sc.keep[i]) {
        a.kept_blk[b0 + runb] = i;
        a.kept_off[b0 + runb] = runb * s.G;
        ++runb;
      }
    if (tid == blockDim.x - 1) a.kept_nblk[r] = runb;
  }
  if (tid == 0) s.kept_count[r] = kept;   // read by the CTA that finishes the batch
  __syncthreads();
  return kept;
}

__global__ void __launch_bounds__(kTailThreads, 1) tail_kernel(const __grid_constant__ TailArgs a) {
  // With the descriptor in the parameters the owned blocks' token ranges come
  // from the parameters alone: worked out while pass 2's last CTAs finish,
  // before the wait for pass 2's partial sums.
  const bool early = a.desc.R > 0;
  pdl_trigger();
  if (!early) pdl_wait();
  extern __shared__ unsigned char s_dyn[];
  __shared__ int s_bstart[kTailMaxBpc + 1];   // first packed token of each owned block, then the run's end
  __shared__ float s_inv[kTailMaxBpc];
  __shared__ int s_sel[kTailMaxBpc];
  __shared__ int s_nsel, s_last;
  const SelectArgs& s = a.s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const DescView dv = tail_view(a);
  const int nb_total = dv.blk[s.R];   // 0 if the describe kernel rejected the descriptor
  if (nb_total == 0) {
    if (early) pdl_wait();
    if (blockIdx.x == 0) finish_batch(a, dv, true);
    return;
  }
  const int b0 = blockIdx.x * a.bpc;
  if (b0 >= nb_total) return;
  const int b1 = min(nb_total, b0 + a.bpc);
  const int nown = b1 - b0;
  // Token ranges of the owned blocks (consecutive blocks are consecutive
  // tokens of the packed batch) and each block's 1/(H_q n_eff).
  if (tid <= nown) {
    const int b = b0 + min(tid, nown - 1);
    const int r = owner_of(dv.blk, s.R, b);
    const int i = b - dv.blk[r];
    const int tok0 = dv.cu[r], L = dv.cu[r + 1] - tok0;
    if (tid < nown) {
      s_bstart[tid] = tok0 + i * s.G;
      s_inv[tid] = 1.0f / float(s.Hq * min(s.n, L));
    } else {
      s_bstart[nown] = tok0 + min(L, (i + 1) * s.G);
    }
  }
  if (tid == 0) {
    s_nsel = 0;
    s_last = 0;
  }
  if (early) pdl_wait();
  __syncthreads();
  const int tfirst = s_bstart[0], ntok = s_bstart[nown] - tfirst;
  float* s_val = reinterpret_cast<float*>(s_dyn);   // [ntok] token scores of the run
  for (int j = tid; j < ntok; j += blockDim.x) {
    const int t = tfirst + j;
    float v;
    if (s.P > 0) {
      int k = 0, hi = nown - 1;   // owned block of token t: the last k with s_bstart[k] <= t
      while (k < hi) {
        const int mid = (k + hi + 1) >> 1;
        if (s_bstart[mid] <= t) k = mid;
        else hi = mid - 1;
      }
      v = 0.f;
#pragma unroll 8
      for (int c = 0; c < s.P; ++c) v += s.part[(int64_t)c * s.T + t];
      v *= s_inv[k];
      if (s.scores_out) s.scores_out[t] = v;
    } else {
      v = s.scores_in[t];
    }
    s_val[j] = v;
  }
  __syncthreads();
  for (int k = warp; k < nown; k += kTailWarps) {
    const int lo = s_bstart[k] - tfirst, hi = s_bstart[k + 1] - tfirst;
    float sum = 0.f;
    for (int j = lo + lane; j < hi; j += 32) sum += s_val[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s.block_scores[b0 + k] = sum / float(hi - lo);   // read by the selecting CTA
  }
  __syncthreads();
  // Count this CTA done on every request its run touches; keep the ones it
  // completes.  The acquire-release increments publish this CTA's block means
  // and, for the CTA that completes a request, make every other CTA's visible.
  if (tid == 0) {
    const int r_first = owner_of(dv.blk, s.R, b0), r_last = owner_of(dv.blk, s.R, b1 - 1);
    int nsel = 0;
    for (int r = r_first; r <= r_last; ++r) {
      const int f = dv.blk[r], e = dv.blk[r + 1];
      if (e == f) continue;   // empty request (no blocks)
      const int ctas = (e - 1) / a.bpc - f / a.bpc + 1;
      if (ctas == 1 || add_acq_rel(a.counters + r, 1) == ctas - 1) s_sel[nsel++] = r;
    }
    s_nsel = nsel;
  }
  __syncthreads();
  const int nsel = s_nsel;
  if (nsel == 0) return;
  const SelectScratch sc = carve_select(s_dyn, a.nbp);
  int kept = 0;
  for (int k = 0; k < nsel; ++k) kept = select_and_emit(a, dv, s_sel[k], sc);
  if (s.R == 1) {
    // One request: its words are all its own (written above), so the batch's
    // offsets and total follow from its count with no further reads.
    if (tid == 0 && a.cu_out) {
      a.cu_out[0] = 0;
      a.cu_out[1] = kept;
      *a.total_kept = kept;
    }
    return;
  }
  if (tid == 0) {
    // With one request (or this CTA completing all of them) nothing else is pending.
    if (nsel == a.nonempty || add_acq_rel(a.counters + s.R, nsel) + nsel == a.nonempty) s_last = 1;
  }
  __syncthreads();
  if (s_last) finish_batch(a, dv, false);
}

// The gather of the fused path: output row o belongs to the request r with
// cu_out[r] <= o < cu_out[r+1]; its kept block is the last one of r's list
// whose output offset is <= o - cu_out[r], and its input row follows from the
// block's first token.  One warp per output row (two, each copying a
// part, when there are fewer rows than warps); block 0 appends the
// drop-history record.
//
// Latency is the cost here (about one row per warp at the usual kept
// fractions), so the dependent round trips are few: warp 0 of each CTA loads
// the total, request 0's kept-block count and request 0's first 32 kept blocks
// at once (its block range is known before the tail's results are), and a
// row of request 0 with at most 32 kept blocks (every row of a single
// request at those fractions) finds its block in shared memory.  Each lane
// then loads all of its row's 16-byte vectors (up to 16, 8 KB a row) before
// it stores any.
constexpr int kGatherThreads = 256;
constexpr int kGatherVec = 16;   // vectors per lane in flight

__global__ void __launch_bounds__(kGatherThreads) gather_list_kernel(const __grid_constant__ GatherListArgs g) {
  __shared__ int s_total, s_nblk0;
  __shared__ int s_off0[32], s_blk0[32];
  if (threadIdx.x == 0) {   // an empty batch: no rows
    s_total = 0;
    s_nblk0 = 0;
  }
  pdl_trigger();
  const CompactArgs& a = g.c;
  const int lane = threadIdx.x & 31;
  // With the descriptor in the parameters, the prologue's addresses come from
  // the parameters alone and are worked out before the wait for the tail.
  const bool early = g.desc.R > 0;
  const int32_t *p_off = nullptr, *p_blk = nullptr;
  if (early && threadIdx.x < 32 && lane < g.desc.blk[1] - g.desc.blk[0]) {
    p_off = g.kept_off + g.desc.blk[0] + lane;
    p_blk = g.kept_blk + g.desc.blk[0] + lane;
  }
  const int32_t* p_total = a.total_kept;
  const int32_t* p_nblk0 = g.kept_nblk;
  pdl_wait();
  const DescView dv = gather_view(g);
  if (threadIdx.x < 32 && a.R > 0) {
    if (!early) {
      const int base0 = dv.blk[0], nb0 = dv.blk[1] - base0;
      if (lane < nb0) {   // inside request 0's block range; entries past its count are unused
        p_off = g.kept_off + base0 + lane;
        p_blk = g.kept_blk + base0 + lane;
      }
    }
    int off = INT_MAX, blk = 0;
    if (p_off) {
      off = *p_off;
      blk = *p_blk;
    }
    const int total = *p_total, nblk0 = *p_nblk0;
    s_off0[lane] = off;
    s_blk0[lane] = blk;
    if (lane == 0) {
      s_total = min(total, a.T);
      s_nblk0 = nblk0;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 32 && a.history) {
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
  __syncthreads();
  const int total = s_total, nblk0 = s_nblk0;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int64_t nvec = a.row_bytes / 16;
  // With fewer rows than warps, two warps share a row (each copies a
  // contiguous part), so the copies spread over more SMs.
  const int wpr = total > 0 ? max(1, min(2, nwarps / total)) : 1;
  const int64_t part_vec = ((nvec + wpr - 1) / wpr + 31) & ~int64_t(31);
  for (int wi = warp; wi < total * wpr; wi += nwarps) {
    const int o = wi / wpr, part = wi - o * wpr;
    const int r = a.R == 1 ? 0 : owner_of(a.cu_out, a.R, o);
    const int j = r == 0 ? o : o - a.cu_out[r];
    const int base = dv.blk[r];
    int lo = 0, n = r == 0 ? nblk0 : g.kept_nblk[r];
    if (n <= 0) continue;   // never for a consistent batch
    int kb = -1, koff = 0;
    if (r == 0 && n <= 32) {
      const int off = lane < n ? s_off0[lane] : INT_MAX;
      const unsigned below = __ballot_sync(0xffffffffu, off <= j);   // lane 0 always: offset 0 <= j
      if (!below) continue;   // never for a consistent batch
      const int last = 31 - __clz(below);
      kb = s_blk0[last];
      koff = s_off0[last];
      n = 1;
    }
    // 32-way search: each lane probes one of 32 evenly spaced kept blocks and
    // the last probe at or below j narrows the range (one round for up to 32
    // kept blocks, two for up to 1024).  Each probe also loads its block's
    // index, so when the probes are single blocks the answer is already in a
    // lane's registers.
    while (n > 1) {
      const int step = (n + 31) >> 5;
      const int at = lane * step;
      int off = INT_MAX, blk = 0;
      if (at < n) {
        off = g.kept_off[base + lo + at];
        blk = g.kept_blk[base + lo + at];
      }
      const unsigned below = __ballot_sync(0xffffffffu, off <= j);   // lane 0 always: offset 0 <= j
      if (!below) break;   // never for a consistent batch
      const int last = 31 - __clz(below);
      lo += last * step;
      n = min(step, n - last * step);
      if (step == 1) {   // the probes were the blocks themselves
        kb = __shfl_sync(0xffffffffu, blk, last);
        koff = __shfl_sync(0xffffffffu, off, last);
      }
    }
    if (n != 1) continue;
    if (kb < 0) {   // one kept block, or the search ended on a range of blocks
      kb = g.kept_blk[base + lo];
      koff = g.kept_off[base + lo];
    }
    const int t = dv.cu[r] + kb * g.G + (j - koff);
    if (t < dv.cu[r] || t >= dv.cu[r + 1] || t >= a.T) continue;   // never for a consistent batch
    const bool first = part == 0;   // the part that writes the row's index, position and slot
    if (first && lane == 0 && a.kept_index) a.kept_index[o] = t;
    // The row's position and slot load with the row itself (lanes 1 and 2).
    int64_t side = 0;
    if (first && lane == 1 && a.pos_in) side = a.pos_in[t];
    if (first && lane == 2 && a.slot_in) side = a.slot_in[t];
    if (a.hidden_in) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.hidden_in) + (int64_t)t * a.row_bytes);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.hidden_out) + (int64_t)o * a.row_bytes);
      const int64_t v_end = min(nvec, (part + 1) * part_vec);
      for (int64_t v0 = part * part_vec + lane; v0 < v_end; v0 += 32 * kGatherVec) {
        uint4 x[kGatherVec];
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u)
          if (v0 + 32 * u < v_end) x[u] = __ldcs(src + v0 + 32 * u);
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u)
          if (v0 + 32 * u < v_end) __stcs(dst + v0 + 32 * u, x[u]);
      }
    }
    if (first && lane == 1 && a.pos_in) a.pos_out[o] = side;
    if (first && lane == 2 && a.slot_in) a.slot_out[o] = side;
  }
}

}  // namespace

static_assert(sizeof(TailArgs) <= 4096 && sizeof(GatherListArgs) <= 4096, "tail kernel parameters within 4 KB");

int tail_blocks_per_cta(int G) {
  int bpc = G > 0 ? kTailThreads / G : 1;   // about one token per thread in the finalize phase
  return bpc < 1 ? 1 : (bpc > kTailMaxBpc ? kTailMaxBpc : bpc);
}

size_t tail_smem_bytes(int G, int max_nb) {
  const int nbp = ((max_nb > 0 ? max_nb : 1) + 7) & ~7;
  const size_t sel = select_smem_bytes(nbp);
  const size_t vals = sizeof(float) * size_t(tail_blocks_per_cta(G)) * size_t(G);
  return sel > vals ? sel : vals;
}

cudaError_t launch_tail(const TailArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = tail_smem_bytes(a.s.G, a.s.max_nb);
  cudaError_t e = cudaFuncSetAttribute(tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int grid = a.s.NB > 0 ? (a.s.NB + a.bpc - 1) / a.bpc : 1;
  return launch_kernel(tail_kernel, grid, kTailThreads, smem, s, pdl, a);
}

cudaError_t launch_gather_list(const GatherListArgs& a, cudaStream_t s, bool pdl) {
  // At most one row per warp, and no more CTAs than fit on the GPU at once
  // (two per SM at this kernel's register count), so the CTAs left without
  // a row finish in the same wave as the others.
  const int wpc = kGatherThreads / 32;
  int blocks = (a.c.T + wpc - 1) / wpc;
  blocks = blocks < 1 ? 1 : (blocks > 2 * kPlanSMs ? 2 * kPlanSMs : blocks);
  return launch_kernel(gather_list_kernel, blocks, kGatherThreads, 0, s, pdl, a);
}

}  // namespace upf
