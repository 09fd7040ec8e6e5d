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
                                                                  MaskParams mp, int B, int nQ,
                                                                  int nK, int nP, int bm,
                                                                  int force_partial) {
  const int e = blockIdx.x;
  const int bb = e / nP;  // batch of this entry (0 when the mask is batch-independent)
  const int p = e % nP;
  char* base = reinterpret_cast<char*>(hdr_out);
  // offsets as in block_mask_geom()
  size_t order_off = (sizeof(BlockMaskHeader) + 15) / 16 * 16;
  size_t cnt_off = (order_off + sizeof(int32_t) * (size_t)bm * nP + 15) / 16 * 16;
  size_t list_off = (cnt_off + sizeof(int32_t) * (size_t)bm * nP + 15) / 16 * 16;
  int32_t* cnt = reinterpret_cast<int32_t*>(base + cnt_off);
  uint32_t* list = reinterpret_cast<uint32_t*>(base + list_off) + (size_t)e * nK;

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
  (void)B;
}

// order[]: entries sorted by descending count (ties by entry index), so the
// heaviest work is scheduled first.  Block 0 also fills the header.
__global__ void __launch_bounds__(kBuildThreads) order_kernel(BlockMaskHeader* hdr, int B,
                                                              MaskParams mp, int nQ, int nK,
                                                              int nP, int bm, int force_partial) {
  const int n = bm * nP;
  char* base = reinterpret_cast<char*>(hdr);
  size_t order_off = (sizeof(BlockMaskHeader) + 15) / 16 * 16;
  size_t cnt_off = (order_off + sizeof(int32_t) * (size_t)n + 15) / 16 * 16;
  size_t list_off = (cnt_off + sizeof(int32_t) * (size_t)n + 15) / 16 * 16;
  int32_t* order = reinterpret_cast<int32_t*>(base + order_off);
  const int32_t* cnt = reinterpret_cast<const int32_t*>(base + cnt_off);

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
    h.order_off = order_off;
    h.cnt_off = cnt_off;
    h.list_off = list_off;
    h.total_bytes = (list_off + sizeof(uint32_t) * (size_t)n * nK + 15) / 16 * 16;
    *hdr = h;
  }
}

}  // namespace

cudaError_t launch_build_block_mask(int B, int S_q, int S_k, const MaskParams& mp,
                                    int force_partial, void* dst, cudaStream_t stream) {
  BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mp.flags);
  BlockMaskHeader* hdr = reinterpret_cast<BlockMaskHeader*>(dst);
  classify_kernel<<<g.n_entries, kBuildThreads, 0, stream>>>(hdr, mp, B, g.nQ, g.nK, g.nP, g.bm,
                                                             force_partial);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int blocks = (g.n_entries + kBuildThreads - 1) / kBuildThreads;
  order_kernel<<<blocks, kBuildThreads, 0, stream>>>(hdr, B, mp, g.nQ, g.nK, g.nP, g.bm,
                                                     force_partial);
  return cudaGetLastError();
}

}  // namespace attn
