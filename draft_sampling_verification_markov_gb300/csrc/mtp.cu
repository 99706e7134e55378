// mtp.cu -- MTP/NextN greedy proposal and greedy verification in two chained launches.
//
// "Module deepseek_v4_mtp", Forward: without a Markov head the draft token of position k is the
// argmax of the draft logits of position k - 1, so the gamma positions do not depend on one
// another. "DeepSeek-V4 MTP/NextN 怎样逐步生成候选", sections 三 and 四: the verify window is
// [bonus, d1 .. d_gamma]; the accepted length is the longest prefix whose drafts equal the
// target argmax of the row before them, and one more target argmax is emitted after it.
//
// Every argmax the step needs (R*gamma draft rows and R*(gamma+1) target rows) therefore comes
// from one pass over the logits. The work items are kMtpChunk-element chunks of those rows, in
// request order (each request's draft rows, then its target rows), and every warp of the
// streaming launch takes a contiguous run of items: its lanes read four 16-byte words per batch
// with the next batch in flight, fold them into (max, first index), and at the end of an item
// the warp's lanes merge and one lane writes the item's partial. No block synchronisation and
// no atomics sit on the stream. A second launch, chained to the first, gives each request a
// block that merges its rows' partials in chunk order (ties go to the lowest token id) and runs
// the greedy scan.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct MtpArgs {
  const void* D;             // draft logits [R, gamma, V]
  const void* T;             // target logits [R, gamma + 1, V]
  int R, gamma, V;
  const int32_t* lengths;    // optional [R]
  int32_t* draft_tokens;     // [R, gamma]
  int32_t* accept_len;       // [R]
  int32_t* out_tokens;       // optional [R, gamma + 1]
  int32_t* next_anchor;      // optional [R]
  float* pm;                 // per item: maximum
  int* pi;                   // per item: first index of the maximum
  uint32_t* status;
  int nchunk;                // chunks per row
  long long items;           // R * (2 gamma + 1) * nchunk
};

// (value, index) with the larger value, the lower index on equal values.
__device__ __forceinline__ void amax_merge(float& m, int& i, float m2, int i2) {
  if (m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_amax(float& m, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
    amax_merge(m, i, m2, i2);
  }
}

// The row (draft or target) and chunk of item q, and whether its words are read at all.
struct Item {
  const char* base;  // first byte of the chunk
  int r;             // request
  int v0;            // first element of the chunk
  int n;             // elements in the chunk
  bool live;         // false: a target row past the request's verified length (not read)
};

template <int DT>
__device__ __forceinline__ Item item_of(const MtpArgs& a, long long q) {
  const int rr = 2 * a.gamma + 1;
  const long long row = q / a.nchunk;
  const int c = (int)(q - row * a.nchunk);
  Item it;
  it.r = (int)(row / rr);
  const int k = (int)(row - (long long)it.r * rr);
  it.v0 = c * kMtpChunk;
  it.n = min(kMtpChunk, a.V - it.v0);
  const size_t es = DT == SPEC_BF16 ? 2 : 4;
  size_t off;
  if (k < a.gamma) {
    off = ((size_t)it.r * a.gamma + k) * a.V + it.v0;
    it.base = static_cast<const char*>(a.D) + off * es;
    it.live = true;
  } else {
    const int i = k - a.gamma;
    off = ((size_t)it.r * (a.gamma + 1) + i) * a.V + it.v0;
    it.base = static_cast<const char*>(a.T) + off * es;
    int l = a.gamma;
    if (a.lengths) l = min(max(a.lengths[it.r], 0), a.gamma);
    it.live = i <= l;
  }
  return it;
}

constexpr int kBatch = 4;  // 16-byte words per lane per batch

// Batches (kBatch words per lane, 32 lanes) per item.
template <int DT>
constexpr int batches_per_item() {
  return kMtpChunk / (DT == SPEC_BF16 ? 8 : 4) / (kBatch * 32);
}

// Words of batch bb of an item: word x = bb * 128 + j * 32 + lane (coalesced 512-byte runs).
template <int DT>
__device__ __forceinline__ void load_batch(const Item& it, int bb, int lane, uint4 (&w)[kBatch]) {
  constexpr int EPW = DT == SPEC_BF16 ? 8 : 4;
  const int nw = it.live ? it.n / EPW : 0;
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    const int x = bb * kBatch * 32 + j * 32 + lane;
    w[j] = x < nw ? ld_stream16(it.base + (size_t)x * 16) : make_uint4(0, 0, 0, 0);
  }
}

// Fold a batch into the lane's (max, first index); words in increasing element order.
template <int DT>
__device__ __forceinline__ void fold_batch(const Item& it, int bb, int lane,
                                           const uint4 (&w)[kBatch], float& m, int& idx) {
  constexpr int EPW = DT == SPEC_BF16 ? 8 : 4;
  const int nw = it.live ? it.n / EPW : 0;
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    const int x = bb * kBatch * 32 + j * 32 + lane;
    if (x >= nw) continue;
    float e[8];
    const uint32_t u[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
    if constexpr (DT == SPEC_BF16) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        e[2 * h] = __uint_as_float(u[h] << 16);
        e[2 * h + 1] = __uint_as_float(u[h] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) e[h] = __uint_as_float(u[h]);
    }
    const int v = it.v0 + x * EPW;
#pragma unroll
    for (int h = 0; h < EPW; ++h)
      if (e[h] > m) {  // strict: the first maximum stays; NaN never wins
        m = e[h];
        idx = v + h;
      }
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) mtp_stream_kernel(MtpArgs a) {
  constexpr int BPI = batches_per_item<DT>();
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const long long nwarps = (long long)gridDim.x * kWarps;
  const long long i0 = a.items * gw / nwarps, i1 = a.items * (gw + 1) / nwarps;
  const long long nb = (i1 - i0) * BPI;
  if (nb == 0) return;
  Item it = item_of<DT>(a, i0), itn = it;
  uint4 cur[kBatch], nxt[kBatch];
  load_batch<DT>(it, 0, lane, cur);
  float m = -INFINITY;
  int idx = 0x7fffffff;
  for (long long b = 0; b < nb; ++b) {
    const int bb = (int)(b % BPI);
    if (b + 1 < nb) {
      const int bn = (int)((b + 1) % BPI);
      if (bn == 0) itn = item_of<DT>(a, i0 + (b + 1) / BPI);
      load_batch<DT>(itn, bn, lane, nxt);
    }
    fold_batch<DT>(it, bb, lane, cur, m, idx);
    if (bb == BPI - 1) {
      warp_amax(m, idx);
      if (lane == 0) {
        const long long q = i0 + b / BPI;
        a.pm[q] = m;
        a.pi[q] = idx;
      }
      m = -INFINITY;
      idx = 0x7fffffff;
      it = itn;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) cur[j] = nxt[j];
  }
}

// One block per request: merge each row's chunk partials, then the greedy scan.
__global__ void __launch_bounds__(kThreads) mtp_scan_kernel(MtpArgs a) {
  extern __shared__ int amax_s[];  // 2 gamma + 1 row argmaxes
  grid_dep_wait();                 // the partials come from the streaming launch before
  const int r = blockIdx.x;
  const int rr = 2 * a.gamma + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int l = a.gamma;
  if (a.lengths) l = min(max(a.lengths[r], 0), a.gamma);
  for (int k = warp; k < rr; k += kWarps) {
    const bool live = k < a.gamma || k - a.gamma <= l;
    float m = -INFINITY;
    int idx = 0x7fffffff;
    if (live) {
      const size_t q0 = ((size_t)r * rr + k) * a.nchunk;
      for (int c = lane; c < a.nchunk; c += 32) amax_merge(m, idx, a.pm[q0 + c], a.pi[q0 + c]);
      warp_amax(m, idx);
      if (idx < 0 || idx >= a.V) {  // no finite maximum in the row
        if (lane == 0) atomicOr(a.status, SPEC_DEV_NONFINITE);
        idx = 0;
      }
    }
    if (lane == 0) amax_s[k] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.lengths) {
      const int l0 = a.lengths[r];
      if (l0 < 0 || l0 > a.gamma) atomicOr(a.status, SPEC_DEV_BAD_LENGTH);
    }
    const int* x = amax_s;            // draft tokens
    const int* y = amax_s + a.gamma;  // target argmax of window rows 0 .. gamma
    for (int k = 0; k < a.gamma; ++k) a.draft_tokens[(size_t)r * a.gamma + k] = x[k];
    int n = 0, t = 0;
    for (int i = 0; i <= l; ++i) {
      t = y[i];
      if (i == l || x[i] != t) break;
      n = i + 1;
    }
    a.accept_len[r] = n;
    if (a.out_tokens) {
      int32_t* o = a.out_tokens + (size_t)r * (a.gamma + 1);
      for (int i = 0; i <= a.gamma; ++i) o[i] = i < n ? x[i] : -1;
      o[n] = t;
    }
    if (a.next_anchor) a.next_anchor[r] = t;
  }
}

}  // namespace

bool mtp_greedy_supported(int dtype, int R, int gamma, int V, const void* D, const void* T) {
  if (R < 1 || gamma < 0 || gamma > kMtpMaxGamma) return false;
  const int epw = dtype == SPEC_BF16 ? 8 : 4;
  if (V % epw != 0) return false;  // rows start on 16-byte boundaries
  const uintptr_t mask = 15;
  if ((reinterpret_cast<uintptr_t>(T) & mask) != 0) return false;
  if (gamma > 0 && (reinterpret_cast<uintptr_t>(D) & mask) != 0) return false;
  return true;
}

cudaError_t launch_mtp_greedy(int dtype, const void* D, const void* T, int R, int gamma, int V,
                              const int32_t* lengths, int32_t* draft_tokens, int32_t* accept_len,
                              int32_t* out_tokens, int32_t* next_anchor, float* pm, int* pi,
                              uint32_t* status, cudaStream_t s) {
  MtpArgs a;
  a.D = D;
  a.T = T;
  a.R = R;
  a.gamma = gamma;
  a.V = V;
  a.lengths = lengths;
  a.draft_tokens = draft_tokens;
  a.accept_len = accept_len;
  a.out_tokens = out_tokens;
  a.next_anchor = next_anchor;
  a.pm = pm;
  a.pi = pi;
  a.status = status;
  a.nchunk = (V + kMtpChunk - 1) / kMtpChunk;
  a.items = (long long)R * (2 * gamma + 1) * a.nchunk;
  {
    TraceScope ts(SPEC_KCLASS_STREAM, s);
    // as many blocks as are resident at once; each warp takes a contiguous run of items
    auto k = dtype == SPEC_BF16 ? mtp_stream_kernel<SPEC_BF16> : mtp_stream_kernel<SPEC_F32>;
    static int cached[2] = {0, 0};
    int& per_sm = cached[dtype == SPEC_BF16];
    if (per_sm < 1) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, 0) != cudaSuccess ||
          per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
      }
    }
    const long long warps_needed = a.items;
    const long long cap = (long long)per_sm * num_sms();
    const long long want = (warps_needed + kWarps - 1) / kWarps;
    const int grid = (int)(want < cap ? want : cap);
    k<<<grid, kThreads, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  const size_t smem = (size_t)(2 * gamma + 1) * sizeof(int);
  return launch_kernel(mtp_scan_kernel, dim3(R), dim3(kThreads), smem, s, true, a);
}

}  // namespace spec
