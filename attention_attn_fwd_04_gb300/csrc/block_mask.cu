// block_mask.cu -- build_block_mask: classify every (query tile, key tile)
// pair as EMPTY / PARTIAL / FULL, compact the non-empty key tiles of every
// pair of query tiles, and order the pairs by descending work.
//
// Tiles where no (query, key) pair is visible are skipped entirely; the
// per-element mask runs only on PARTIAL tiles.  This is the block-sparse
// structure behind masks that never materialise the quadratic matrix
// ("PyTorch 2.5 Introduces FlexAttention and TorchDynamo C++ Runtime",
// body; "FlashAttention-4 explained", "PyTorch Gets the Upgrade Too").
//
// Classification is exact for the interval masks (causal, window,
// prefix-LM, the S_k bound) and conservative for documents: a tile is
// EMPTY for documents only when the document-id ranges of its rows and its
// keys do not meet, FULL only when every row and key lies in one document.
// For non-decreasing document ids (packed sequences) both tests are exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {

namespace {

constexpr int kBuildThreads = 256;     // order kernel
constexpr int kClassifyThreads = 256;   // classify kernel: one key tile per thread

struct Range {
  int lo, hi;
};

// Visible key interval [lo, hi] of query row i from the interval masks
// (pl: the batch's prefix length).  64-bit, so no window or offset overflows.
__device__ __forceinline__ void row_interval(long long i, long long pl, const MaskParams& mp,
                                             long long& lo, long long& hi) {
  const long long qpos = i + mp.q_offset;
  lo = 0;
  hi = mp.S_k - 1;
  if (mp.flags & ATTN_MASK_CAUSAL) hi = min(hi, qpos);
  if (mp.flags & ATTN_MASK_WINDOW) {
    lo = max(lo, qpos - mp.window + 1);
    hi = min(hi, qpos);
  }
  if (mp.flags & ATTN_MASK_PREFIX_LM) hi = min(hi, max(qpos, pl - 1));
}

__device__ __forceinline__ bool row_meets(long long i, long long pl, int c0, int c1,
                                          const MaskParams& mp) {
  long long lo, hi;
  row_interval(i, pl, mp, lo, hi);
  return max(lo, (long long)c0) <= min(hi, (long long)c1);
}

// Class of (query rows [r0, r1], key tile starting at c0), in O(1).
//
// Every interval mask gives row i a visible key interval [lo(i), hi(i)]
// whose ends never decrease as i grows.  Hence
//  * FULL: all rows see the whole tile  <=>  lo(r1) <= c0 and
//    hi(r0) >= c0 + 127 (and the tile is not cut by S_k);
//  * non-EMPTY: some row meets [c0, c1].  The overlap length
//    min(hi, c1) - max(lo, c0) is piecewise linear in the row with integer
//    breakpoints, so its maximum over [r0, r1] is taken at r0, r1 or a
//    breakpoint: the positions where lo leaves 0 (qpos = W - 1) or passes c0
//    (qpos = c0 + W - 1), where hi reaches S_k - 1, the prefix end
//    (qpos = P - 1) or c1.  Testing those rows is exact.
// Documents (dq/dk: id ranges of the rows and of the keys) are then applied
// conservatively: EMPTY when the ranges do not meet, FULL only when both are
// one and the same document.
// The user block map's verdict on tile (qt, kt) of mask batch bb: false
// hides the whole tile.
__device__ __forceinline__ bool block_open(const MaskParams& mp, int bb, int qt, int kt, int nQ,
                                           int nK) {
  if (!(mp.flags & ATTN_MASK_BLOCKS)) return true;
  const size_t mb = (mp.flags & kMaskBlocksBatched) ? (size_t)bb : 0;
  return mp.blocks[(mb * nQ + qt) * nK + kt] != 0;
}

__device__ uint32_t classify_tile(int r0, int r1, int c0, long long pl, const MaskParams& mp,
                                  Range dq, Range dk) {
  if (r0 > r1) return kEmpty;  // no valid query row
  const int c1 = min(c0 + kTileN - 1, mp.S_k - 1);
  const bool ragged = (c1 - c0 + 1) < kTileN;
  const long long w = (mp.flags & ATTN_MASK_WINDOW) ? mp.window : 1;
  const long long cand[5] = {w - 1, c0 + w - 1, (long long)mp.S_k - 1, pl - 1, c1};
  bool any = row_meets(r0, pl, c0, c1, mp) || row_meets(r1, pl, c0, c1, mp);
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const long long i = min(max(cand[k] - mp.q_offset, (long long)r0), (long long)r1);
    any = any || row_meets(i, pl, c0, c1, mp);
  }
  if (!any) return kEmpty;
  long long lo1, hi1, lo0, hi0;
  row_interval(r1, pl, mp, lo1, hi1);
  row_interval(r0, pl, mp, lo0, hi0);
  bool all = !ragged && lo1 <= c0 && hi0 >= (long long)c0 + kTileN - 1;
  if (mp.flags & ATTN_MASK_DOCUMENT) {
    if (dk.hi < dq.lo || dq.hi < dk.lo) return kEmpty;
    if (!(dq.lo == dq.hi && dk.lo == dk.hi && dq.lo == dk.lo)) all = false;
  }
  return all ? kFull : kPartial;
}

// One block per (batch entry, group of g.tpe query tiles).  Writes cnt[e]
// and the compacted list of key tiles that are non-empty for some query tile
// of the group, in descending key-tile order, one key tile per thread,
// kClassifyThreads tiles at a time.
__global__ void __launch_bounds__(kClassifyThreads) classify_kernel(BlockMaskHeader* hdr_out,
                                                                     MaskParams mp,
                                                                     BlockMaskGeom g,
                                                                     int force_partial) {
  constexpr int kWarps = kClassifyThreads / 32;
  const int nQ = g.nQ, nK = g.nK, nP = g.nP, tpe = g.tpe;
  const int e = blockIdx.x;
  const int bb = e / nP;  // batch of this entry (0 when the mask is batch-independent)
  const int p = e % nP;
  char* base = reinterpret_cast<char*>(hdr_out);
  int32_t* cnt = reinterpret_cast<int32_t*>(base + g.cnt_off);
  uint32_t* list = reinterpret_cast<uint32_t*>(base + g.list_off) + (size_t)e * nK;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  __shared__ int s_warp_cnt[kWarps];
  // DOCUMENT: id range of every key tile of this batch (S_q == S_k, so the
  // query tiles have the same ranges)
  const bool docs = (mp.flags & ATTN_MASK_DOCUMENT) != 0;
  const int32_t* t_lo = docs ? reinterpret_cast<const int32_t*>(base + g.tile_off) + (size_t)bb * nK
                             : nullptr;
  const int32_t* t_hi = docs ? t_lo + (size_t)g.bm * nK : nullptr;
  const long long pl = (mp.flags & ATTN_MASK_PREFIX_LM) ? mp.prefix_len[bb] : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  int r0[kTilesPerQuad], r1[kTilesPerQuad];
  Range dq[kTilesPerQuad];
#pragma unroll
  for (int t = 0; t < kTilesPerQuad; ++t) {
    const int qt = tpe * p + t;
    r0[t] = qt * kTileM;
    r1[t] = (t < tpe && qt < nQ) ? min(r0[t] + kTileM - 1, mp.S_q - 1) : r0[t] - 1;
    dq[t] = (docs && r0[t] <= r1[t]) ? Range{t_lo[qt], t_hi[qt]} : Range{0, 0};
  }

  int total = 0;
  for (int chunk = 0; chunk < nK; chunk += kClassifyThreads) {
    const int idx = chunk + threadIdx.x;  // position in descending key-tile order
    uint32_t entry = 0;
    bool keep = false;
    if (idx < nK) {
      const int kt = nK - 1 - idx;
      const int c0 = kt * kTileN;
      const Range dk = docs ? Range{t_lo[kt], t_hi[kt]} : Range{0, 0};
      entry = (uint32_t)kt;
#pragma unroll
      for (int t = 0; t < kTilesPerQuad; ++t) {
        // rows past the group or past S_q: r1 < r0, classified EMPTY
        uint32_t c = (r0[t] <= r1[t] && block_open(mp, bb, tpe * p + t, kt, nQ, nK))
                         ? classify_tile(r0[t], r1[t], c0, pl, mp, dq[t], dk)
                         : kEmpty;
        if (force_partial && c == kFull) c = kPartial;
        keep |= c != kEmpty;
        entry |= c << (24 + 2 * t);
      }
    }
    // stable compaction within the chunk: warp ballots + block prefix
    const unsigned ball = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_warp_cnt[warp] = __popc(ball);
    __syncthreads();
    int before = 0, chunk_total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += s_warp_cnt[w];
      chunk_total += s_warp_cnt[w];
    }
    before += __popc(ball & ((1u << lane) - 1u));
    if (keep) list[total + before] = entry;
    total += chunk_total;
    __syncthreads();  // s_warp_cnt is reused by the next chunk
  }
  if (threadIdx.x == 0) cnt[e] = total;
}

// One block per (mask batch, key tile) of the transposed mask: the query
// tiles that see some key of the tile, ascending, with their classes (the
// same classifier as the forward's mask, so the two always agree).
__global__ void __launch_bounds__(kClassifyThreads) classify_t_kernel(char* dst_t,
                                                                       const char* fwd_mask,
                                                                       MaskParams mp,
                                                                       BlockMaskGeom g,
                                                                       BlockMaskTGeom gt,
                                                                       int force_partial) {
  constexpr int kWarps = kClassifyThreads / 32;
  const int e = blockIdx.x;
  const int bb = e / gt.nK, kt = e % gt.nK;
  int32_t* cnt = reinterpret_cast<int32_t*>(dst_t);
  uint32_t* list = reinterpret_cast<uint32_t*>(dst_t + gt.list_off) + (size_t)e * gt.nQ;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  __shared__ int s_warp_cnt[kWarps];
  const bool docs = (mp.flags & ATTN_MASK_DOCUMENT) != 0;
  const int32_t* t_lo =
      docs ? reinterpret_cast<const int32_t*>(fwd_mask + g.tile_off) + (size_t)bb * g.nK : nullptr;
  const int32_t* t_hi = docs ? t_lo + (size_t)g.bm * g.nK : nullptr;
  const long long pl = (mp.flags & ATTN_MASK_PREFIX_LM) ? mp.prefix_len[bb] : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = kt * kTileN;
  const Range dk = docs ? Range{t_lo[kt], t_hi[kt]} : Range{0, 0};
  int total = 0;
  for (int chunk = 0; chunk < gt.nQ; chunk += kClassifyThreads) {
    const int qt = chunk + threadIdx.x;
    uint32_t entry = 0;
    bool keep = false;
    if (qt < gt.nQ) {
      const int r0 = qt * kTileM, r1 = min(r0 + kTileM - 1, mp.S_q - 1);
      const Range dq = docs ? Range{t_lo[qt], t_hi[qt]} : Range{0, 0};
      uint32_t c = block_open(mp, bb, qt, kt, gt.nQ, gt.nK)
                       ? classify_tile(r0, r1, c0, pl, mp, dq, dk)
                       : kEmpty;
      if (force_partial && c == kFull) c = kPartial;
      keep = c != kEmpty;
      entry = (uint32_t)qt | (c << 24);
    }
    const unsigned ball = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_warp_cnt[warp] = __popc(ball);
    __syncthreads();
    int before = 0, chunk_total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += s_warp_cnt[w];
      chunk_total += s_warp_cnt[w];
    }
    before += __popc(ball & ((1u << lane) - 1u));
    if (keep) list[total + before] = entry;
    total += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) cnt[e] = total;
}

// First position pos in [lo, hi) with row[pos] > v (strict) or row[pos] >= v,
// for ids that are non-decreasing on [lo, hi); hi when there is none.  The
// warp probes 32 evenly spaced positions per step, so a step shrinks the
// range 32-fold.  Every lane returns the result.  Positions stay in [lo, hi)
// whatever the ids.
__device__ int warp_search(const int32_t* row, int lo, int hi, int32_t v, bool strict, int lane) {
  while (hi > lo) {
    const long long len = hi - lo;
    const int p = (len <= 32) ? lo + min(lane, (int)len - 1)
                              : lo + (int)(((long long)(lane + 1) * len) / 32) - 1;
    const int32_t x = row[p];
    const bool pred = (len <= 32 && lane >= len) ? false : (strict ? x > v : x >= v);
    const unsigned m = __ballot_sync(0xffffffffu, pred);
    if (m == 0) return hi;
    const int f = __ffs(m) - 1;
    const int pf = __shfl_sync(0xffffffffu, p, f);
    if (len <= 32) return pf;
    const int prev = __shfl_sync(0xffffffffu, p, f == 0 ? 0 : f - 1);
    hi = pf + 1;
    lo = (f == 0) ? lo : prev + 1;
    if (hi - lo == 1) return lo;  // pred holds at pf and not at pf - 1
  }
  return hi;
}

__global__ void __launch_bounds__(kDocPrepTokens) doc_prep_kernel(const int32_t* ids, int S,
                                                                   char* base, BlockMaskGeom g) {
  constexpr int kWarps = kDocPrepTokens / 32;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int b = blockIdx.y;
  const int i0 = blockIdx.x * kDocPrepTokens;
  const int i = i0 + threadIdx.x;
  const int last = min(i0 + kDocPrepTokens, S) - 1;  // last token of this block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t* row = ids + (size_t)b * S;
  const bool in = i < S;
  const int32_t x = in ? row[i] : 0;
  const bool starts = in && (i == 0 || row[i - 1] != x);
  const bool ends = in && (i == S - 1 || row[i + 1] != x);
  const bool disorder = in && i + 1 < S && row[i + 1] < x;

  __shared__ int s_start[kWarps], s_end[kWarps], s_tmin[kWarps], s_tmax[kWarps];
  __shared__ int s_edge_lo, s_edge_hi;
  // start of the run holding token i0 / end of the run holding token `last`
  // (warp 0 / warp 1, 32-way searches)
  if (warp == 0) {
    const int32_t v = row[i0];
    const int pos = warp_search(row, 0, i0, v, false, lane);  // first row[pos] >= v
    if (lane == 0) s_edge_lo = pos;
  } else if (warp == 1) {
    const int32_t v = row[last];
    const int pos = warp_search(row, last + 1, S, v, true, lane);  // first row[pos] > v
    if (lane == 0) s_edge_hi = pos - 1;
  }
  // inclusive max-scan of run starts, inclusive suffix min-scan of run ends
  int st = starts ? i : -1, en = ends ? i : INT32_MAX;
  int32_t tmin = in ? x : INT32_MAX, tmax = in ? x : INT32_MIN;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, st, o);
    const int d = __shfl_down_sync(0xffffffffu, en, o);
    if (lane >= o) st = max(st, u);
    if (lane + o < 32) en = min(en, d);
    tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  }
  if (lane == 31) s_start[warp] = st;
  if (lane == 0) {
    s_end[warp] = en;
    s_tmin[warp] = tmin;
    s_tmax[warp] = tmax;
  }
  const int any_disorder = __syncthreads_or(disorder);
  for (int w = 0; w < warp; ++w) st = max(st, s_start[w]);
  for (int w = warp + 1; w < kWarps; ++w) en = min(en, s_end[w]);
  if (in) {
    int32_t* dlo = reinterpret_cast<int32_t*>(base + g.doc_off) + (size_t)b * S;
    int32_t* dhi = reinterpret_cast<int32_t*>(base + g.doc_off) + ((size_t)g.bm + b) * S;
    dlo[i] = st >= 0 ? st : s_edge_lo;
    dhi[i] = en != INT32_MAX ? en : s_edge_hi;
  }
  constexpr int kTilesPerBlock = kDocPrepTokens / kTileN;
  constexpr int kWarpsPerTile = kTileN / 32;
  if (threadIdx.x < kTilesPerBlock) {
    const int t = threadIdx.x;
    if (i0 + t * kTileN < S) {
      int32_t lo = INT32_MAX, hi = INT32_MIN;
      for (int w = t * kWarpsPerTile; w < (t + 1) * kWarpsPerTile; ++w) {
        lo = min(lo, s_tmin[w]);
        hi = max(hi, s_tmax[w]);
      }
      const int kt = i0 / kTileN + t;
      int32_t* tl = reinterpret_cast<int32_t*>(base + g.tile_off);
      tl[(size_t)b * g.nK + kt] = lo;
      tl[((size_t)g.bm + b) * g.nK + kt] = hi;
    }
  }
  if (threadIdx.x == 0)
    reinterpret_cast<int32_t*>(base + g.flag_off)[b * gridDim.x + blockIdx.x] = any_disorder;
}

// order[]: entries sorted by descending count (ties by entry index), so the
// heaviest work is scheduled first.  Block 0 also fills the header.
__global__ void __launch_bounds__(kBuildThreads) order_kernel(BlockMaskHeader* hdr, int B,
                                                              MaskParams mp, BlockMaskGeom g,
                                                              int force_partial) {
  const int nQ = g.nQ, nK = g.nK, nP = g.nP, bm = g.bm;
  const int n = bm * nP;
  char* base = reinterpret_cast<char*>(hdr);
  int32_t* order = reinterpret_cast<int32_t*>(base + g.order_off);
  const int32_t* cnt = reinterpret_cast<const int32_t*>(base + g.cnt_off);

  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  int disorder = 0;  // block 0: any document prep block saw ids out of order
  if (blockIdx.x == 0) {
    const int32_t* flags = reinterpret_cast<const int32_t*>(base + g.flag_off);
    for (int j = threadIdx.x; j < g.n_flags; j += kBuildThreads) disorder |= flags[j];
    disorder = __syncthreads_or(disorder);
  }
  __shared__ int s_cnt[kBuildThreads];
  int mine = (e < n) ? cnt[e] : 0;
  int rank = 0;
  int mn = INT32_MAX, mx = INT32_MIN;
  for (int c = 0; c < n; c += kBuildThreads) {
    __syncthreads();
    if (c + threadIdx.x < n) s_cnt[threadIdx.x] = cnt[c + threadIdx.x];
    __syncthreads();
    int lim = min(kBuildThreads, n - c);
    for (int t = 0; t < lim; ++t) {
      int o = s_cnt[t];
      int oe = c + t;
      rank += (o > mine) || (o == mine && oe < e);
      mn = min(mn, o);
      mx = max(mx, o);
    }
  }
  if (e < n) order[rank] = e;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    BlockMaskHeader h;
    h.magic = kBlockMaskMagic;
    h.version = kBlockMaskVersion;
    h.B = B;
    h.S_q = mp.S_q;
    h.S_k = mp.S_k;
    h.nQ = nQ;
    h.nK = nK;
    h.nP = nP;
    h.bm = bm;
    h.n_entries = n;
    h.mask_flags = mp.flags;
    h.window = mp.window;
    h.q_offset = mp.q_offset;
    h.force_partial = force_partial;
    h.uniform = (mn == mx) ? 1 : 0;
    h.max_cnt = mx;
    h.doc_ptr = reinterpret_cast<uint64_t>(mp.doc_ids);
    h.prefix_ptr = reinterpret_cast<uint64_t>(mp.prefix_len);
    h.order_off = g.order_off;
    h.cnt_off = g.cnt_off;
    h.list_off = g.list_off;
    h.total_bytes = g.total;
    h.doc_off = g.doc_off;
    h.docs_sorted = (g.flag_off != 0 && !disorder) ? 1 : 0;
    h.tiles_per_entry = g.tpe;
    h.blocks_ptr = reinterpret_cast<uint64_t>(mp.blocks);
    h.pad2_ = 0;
    *hdr = h;
  }
}

// Every kernel of the build waits for its predecessor in the stream before
// touching memory and is launched with programmatic stream serialization, so
// its launch overlaps the tail of the kernel before it.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, int threads, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_build_block_mask(int B, int S_q, int S_k, const MaskParams& mp,
                                    int force_partial, void* dst, cudaStream_t stream, int tpe) {
  BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mp.flags, tpe);
  BlockMaskHeader* hdr = reinterpret_cast<BlockMaskHeader*>(dst);
  char* base = reinterpret_cast<char*>(dst);
  cudaError_t err;
  if (g.flag_off != 0) {
    const dim3 grid((unsigned)((S_k + kDocPrepTokens - 1) / kDocPrepTokens), (unsigned)g.bm, 1);
    err = launch_pdl(doc_prep_kernel, grid, kDocPrepTokens, stream,
                     static_cast<const int32_t*>(mp.doc_ids), S_k, base, g);
    if (err != cudaSuccess) return err;
  }
  err = launch_pdl(classify_kernel, dim3((unsigned)g.n_entries), kClassifyThreads, stream, hdr, mp,
                   g, force_partial);
  if (err != cudaSuccess) return err;
  const int blocks = (g.n_entries + kBuildThreads - 1) / kBuildThreads;
  return launch_pdl(order_kernel, dim3((unsigned)blocks), kBuildThreads, stream, hdr, B, mp, g,
                    force_partial);
}

cudaError_t launch_build_block_mask_t(int B, int S_q, int S_k, const MaskParams& mp,
                                      int force_partial, const void* fwd_mask, void* dst_t,
                                      cudaStream_t stream) {
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mp.flags);
  const BlockMaskTGeom gt = block_mask_t_geom(B, S_q, S_k, mp.flags);
  return launch_pdl(classify_t_kernel, dim3((unsigned)gt.n_entries), kClassifyThreads, stream,
                    static_cast<char*>(dst_t), static_cast<const char*>(fwd_mask), mp, g, gt,
                    force_partial);
}

}  // namespace attn
