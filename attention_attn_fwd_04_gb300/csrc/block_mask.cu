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

namespace attn {

namespace {

constexpr int kBuildThreads = 256;

struct Range {
  int lo, hi;
};

// Visible key interval [lo, hi] of query row i from the interval masks.
__device__ __forceinline__ Range row_interval(int i, int b, const MaskParams& mp) {
  int qpos = i + mp.q_offset;
  int lo = 0, hi = mp.S_k - 1;
  if (mp.flags & ATTN_MASK_CAUSAL) hi = min(hi, qpos);
  if (mp.flags & ATTN_MASK_WINDOW) {
    lo = max(lo, qpos - mp.window + 1);
    hi = min(hi, qpos);
  }
  if (mp.flags & ATTN_MASK_PREFIX_LM) hi = min(hi, max(qpos, mp.prefix_len[b] - 1));
  return Range{lo, hi};
}

// Class of (query rows [r0, r1], key tile starting at c0) for batch b.
// dq/dk: document-id ranges of the rows and of the keys (DOCUMENT only).
__device__ uint32_t classify(int r0, int r1, int c0, int b, const MaskParams& mp, Range dq,
                             Range dk) {
  if (r0 > r1) return kEmpty;  // no valid query row
  const int c1 = min(c0 + kTileN - 1, mp.S_k - 1);
  const bool ragged = (c1 - c0 + 1) < kTileN;
  bool any = false, all = !ragged;
  for (int i = r0; i <= r1; ++i) {
    Range r = row_interval(i, b, mp);
    int a = max(r.lo, c0), e = min(r.hi, c1);
    if (e >= a) {
      any = true;
      if (a != c0 || e != c0 + kTileN - 1) all = false;
    } else {
      all = false;
    }
  }
  if (!any) return kEmpty;
  if (mp.flags & ATTN_MASK_DOCUMENT) {
    if (dk.hi < dq.lo || dq.hi < dk.lo) return kEmpty;
    if (!(dq.lo == dq.hi && dk.lo == dk.hi && dq.lo == dk.lo)) all = false;
  }
  return all ? kFull : kPartial;
}

__device__ Range doc_range(const int32_t* ids, int a, int e) {
  Range r{INT32_MAX, INT32_MIN};
  for (int j = a; j <= e; ++j) {
    int d = ids[j];
    r.lo = min(r.lo, d);
    r.hi = max(r.hi, d);
  }
  return r;
}

// One block per (batch entry, query-tile pair).  Writes cnt[e] and the
// compacted list of non-empty key tiles in descending key-tile order.
__global__ void __launch_bounds__(kBuildThreads) classify_kernel(BlockMaskHeader* hdr_out,
                                                                  MaskParams mp, BlockMaskGeom g,
                                                                  int force_partial) {
  const int nQ = g.nQ, nK = g.nK, nP = g.nP;
  const int e = blockIdx.x;
  const int bb = e / nP;  // batch of this entry (0 when the mask is batch-independent)
  const int p = e % nP;
  char* base = reinterpret_cast<char*>(hdr_out);
  int32_t* cnt = reinterpret_cast<int32_t*>(base + g.cnt_off);
  uint32_t* list = reinterpret_cast<uint32_t*>(base + g.list_off) + (size_t)e * nK;
  if (e == 0 && threadIdx.x == 0 && g.flag_off != 0)
    *reinterpret_cast<int32_t*>(base + g.flag_off) = 0;  // set by doc_ranges_kernel

  __shared__ Range s_dq[2];
  __shared__ int s_total;
  __shared__ int s_warp_cnt[kBuildThreads / 32];
  const int* ids = (mp.flags & ATTN_MASK_DOCUMENT) ? mp.doc_ids + (size_t)bb * mp.S_k : nullptr;

  if (threadIdx.x < 2) {
    int qt = 2 * p + threadIdx.x;
    int r0 = qt * kTileM, r1 = min(r0 + kTileM - 1, mp.S_q - 1);
    s_dq[threadIdx.x] = (ids && r0 <= r1) ? doc_range(ids, r0, r1) : Range{0, 0};
  }
  if (threadIdx.x == 0) s_total = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Process key tiles from the highest index down, one per thread per chunk.
  for (int chunk = 0; chunk < nK; chunk += kBuildThreads) {
    int idx = chunk + threadIdx.x;  // position in descending order
    uint32_t entry = 0;
    bool keep = false;
    if (idx < nK) {
      int kt = nK - 1 - idx;
      int c0 = kt * kTileN;
      Range dk{0, 0};
      if (ids) dk = doc_range(ids, c0, min(c0 + kTileN - 1, mp.S_k - 1));
      uint32_t cls[2];
      for (int t = 0; t < 2; ++t) {
        int qt = 2 * p + t;
        int r0 = qt * kTileM, r1 = min(r0 + kTileM - 1, mp.S_q - 1);
        cls[t] = (qt < nQ) ? classify(r0, r1, c0, bb, mp, s_dq[t], dk) : kEmpty;
        if (force_partial && cls[t] == kFull) cls[t] = kPartial;
      }
      keep = (cls[0] != kEmpty) || (cls[1] != kEmpty);
      entry = list_entry((uint32_t)kt, cls[0], cls[1]);
    }
    // stable compaction within the chunk: warp ballots + block prefix
    unsigned ball = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_warp_cnt[warp] = __popc(ball);
    __syncthreads();
    int before = 0, chunk_total = 0;
    for (int w = 0; w < kBuildThreads / 32; ++w) {
      if (w < warp) before += s_warp_cnt[w];
      chunk_total += s_warp_cnt[w];
    }
    before += __popc(ball & ((1u << lane) - 1u));
    if (keep) list[s_total + before] = entry;
    __syncthreads();
    if (threadIdx.x == 0) s_total += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) cnt[e] = s_total;
}

// For every token of every mask batch: the first and last key of its
// document, by binary search over the ids (meaningful when the ids are
// non-decreasing, i.e. packed documents), and a flag raised when some
// batch's ids are out of order.  With packed ids, "key j is in query i's
// document" is exactly j in [doc_lo[i], doc_hi[i]].
__global__ void __launch_bounds__(kBuildThreads) doc_ranges_kernel(const int32_t* ids, int S,
                                                                    int bm, char* base,
                                                                    BlockMaskGeom g) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)bm * S) return;
  const int b = (int)(idx / S), i = (int)(idx % S);
  const int32_t* row = ids + (size_t)b * S;
  const int32_t x = row[i];
  if (i + 1 < S && row[i + 1] < x) atomicOr(reinterpret_cast<int32_t*>(base + g.flag_off), 1);
  int lo = 0, hi = S;  // first position with row[pos] >= x
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (row[mid] < x) lo = mid + 1; else hi = mid;
  }
  const int first = lo;
  lo = i;
  hi = S;  // first position with row[pos] > x, searching from i
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (row[mid] <= x) lo = mid + 1; else hi = mid;
  }
  int32_t* dlo = reinterpret_cast<int32_t*>(base + g.doc_off);
  dlo[idx] = first;
  dlo[(size_t)bm * S + idx] = lo - 1;
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
    h.docs_sorted =
        (g.flag_off != 0) ? (*reinterpret_cast<const int32_t*>(base + g.flag_off) == 0) : 0;
    h.pad_ = 0;
    *hdr = h;
  }
}

}  // namespace

cudaError_t launch_build_block_mask(int B, int S_q, int S_k, const MaskParams& mp,
                                    int force_partial, void* dst, cudaStream_t stream) {
  BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mp.flags);
  BlockMaskHeader* hdr = reinterpret_cast<BlockMaskHeader*>(dst);
  classify_kernel<<<g.n_entries, kBuildThreads, 0, stream>>>(hdr, mp, g, force_partial);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (g.flag_off != 0) {
    const long long toks = (long long)g.bm * S_k;
    doc_ranges_kernel<<<(unsigned)((toks + kBuildThreads - 1) / kBuildThreads), kBuildThreads, 0,
                        stream>>>(mp.doc_ids, S_k, g.bm, reinterpret_cast<char*>(dst), g);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  int blocks = (g.n_entries + kBuildThreads - 1) / kBuildThreads;
  order_kernel<<<blocks, kBuildThreads, 0, stream>>>(hdr, B, mp, g, force_partial);
  return cudaGetLastError();
}

}  // namespace attn
