// rows.cu -- streaming row reductions, the generic (CUDA-core) Markov producer, and the
// select / verify / finalize consumers of libspecmarkov.
//
// Producers reduce every (row, segment) of a pass to a partial:
//   stream_partials_kernel   rank-0 rows (no Markov bias): a pure HBM stream of 16-byte loads;
//   markov_ffma_partials     rows with a Markov bias computed on CUDA cores in the canonical
//                            fp32 order (fp32 weights, and every shape the tcgen05 kernel does
//                            not take).
// Consumers:
//   select_kernel            per row: combine partials, then greedy argmax or the inverse-CDF
//                            draw (recomputing only the crossing segment);
//   finalize_stats_kernel    per row (m, log Z);
//   greedy_scan_kernel       per request longest-prefix match + bonus;
//   accept_kernel            per request rejection-sampling acceptance scan;
//   tv_finalize_kernel       per request c* and the survival product.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace spec {

// ------------------------------------------------------------------------------ pair values

// Element value of a MODE_RESID / MODE_TV pass at column v.
template <int UDT, int WDT, int MODE>
__device__ __forceinline__ float pair_value(const RowJob& j, const RowInfo& ri, Norm dn, Norm tn,
                                            int v) {
  const float pt = prob_of(target_logit<UDT>(j, ri, v), tn);
  if (MODE == MODE_RESID && !ri.resid) return pt;  // bonus row: q = p_t
  const float pd = prob_of(draft_logit<UDT, WDT>(j, ri, v), dn);
  if (MODE == MODE_RESID) return fmaxf(pt - pd, 0.0f);
  return fminf(pt, pd);
}

__device__ __forceinline__ void row_norms(const RowJob& j, const RowInfo& ri, Norm& dn, Norm& tn) {
  dn = {0.0f, 0.0f};
  tn = {0.0f, 0.0f};
  if (ri.trow >= 0 && j.tstats) tn = load_norm(j.tstats, ri.trow);
  if (ri.urow >= 0 && j.dstats) dn = load_norm(j.dstats, ri.urow);
}

// ------------------------------------------------------------------------------ streaming producer

// 8 consecutive elements starting at v (v % 8 == 0), vectorised when `vec`.
template <int DT>
__device__ __forceinline__ void load8(const void* base, size_t row_off, int v, int V, bool vec,
                                      float (&x)[8]) {
  if constexpr (DT == SPEC_BF16) {
    const unsigned short* p = reinterpret_cast<const unsigned short*>(base) + row_off + v;
    if (vec && v + 8 <= V) {
      const uint4 q = ld_stream16(p);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = (v + i < V) ? bf16_to_f32(__ldg(p + i)) : -INFINITY;
    }
  } else {
    const float* p = reinterpret_cast<const float*>(base) + row_off + v;
    if (vec && v + 8 <= V) {
      const uint4 q0 = ld_stream16(p), q1 = ld_stream16(p + 4);
      x[0] = __uint_as_float(q0.x); x[1] = __uint_as_float(q0.y);
      x[2] = __uint_as_float(q0.z); x[3] = __uint_as_float(q0.w);
      x[4] = __uint_as_float(q1.x); x[5] = __uint_as_float(q1.y);
      x[6] = __uint_as_float(q1.z); x[7] = __uint_as_float(q1.w);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = (v + i < V) ? __ldg(p + i) : -INFINITY;
    }
  }
}

// Rank-0 rows. One block per (row, segment) unit, grid-stride. MODE_STATS reduces the row's
// primary logits (U if the row has a draft side, else the target); SUM / ARGMAX select which
// halves of the partial are needed. MODE_RESID / MODE_TV reduce the pair value. Each thread
// issues kBatch independent 16-byte loads (per tensor) before doing any arithmetic on them.
constexpr int kBatch = 4;

template <int DT, int MODE, bool SUM, bool ARGMAX>
__global__ void __launch_bounds__(256) stream_partials_kernel(RowJob j, int seg, int nseg, bool vec,
                                                              float* pm, float* ps, int* pi) {
  const int units = j.rows * nseg;
  const int step = blockDim.x * 8;  // columns per block-wide vector sweep
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int row = u / nseg, sg = u - row * nseg;
    const RowInfo ri = row_info(j, row);
    const int v0 = sg * seg, v1 = min(j.V, v0 + seg);
    const size_t out = (size_t)row * nseg + sg;
    if (!ri.active) {
      if (threadIdx.x == 0) {
        if (pm) pm[out] = -INFINITY;
        if (ps) ps[out] = 0.0f;
        if (pi) pi[out] = 0x7fffffff;
      }
      continue;
    }
    if constexpr (MODE == MODE_STATS) {
      const bool draft = ri.urow >= 0;
      const void* src = draft ? j.U : j.T;
      const size_t off = (size_t)(draft ? ri.urow : ri.trow) * j.V;
      StatsAcc acc = stats_empty();
      for (int base = v0 + threadIdx.x * 8; base < v1; base += kBatch * step) {
        float x[kBatch][8];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) load8<DT>(src, off, base + b * step, v1, vec, x[b]);
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = base + b * step;
          float g = -INFINITY;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[b][i] = __fmul_rn(x[b][i], j.scale);
            if (draft && j.mask && !draft_allowed(j, ri.r, v + i)) x[b][i] = -INFINITY;
            if (ARGMAX && x[b][i] > acc.m && x[b][i] > g) acc.idx = v + i;  // first maximum
            g = fmaxf(g, x[b][i]);
          }
          if (g > acc.m) {
            if (SUM && acc.s != 0.0f) acc.s *= exp_shift(acc.m, g);
            acc.m = g;
          }
          if (SUM && acc.m != -INFINITY) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc.s += exp_shift(x[b][i], acc.m);
          }
        }
      }
      acc = block_merge(acc);
      if (threadIdx.x == 0) {
        pm[out] = acc.m;
        if (ps) ps[out] = acc.s;
        if (pi) pi[out] = acc.idx;
      }
    } else {
      Norm dn, tn;
      row_norms(j, ri, dn, tn);
      const bool pair = MODE == MODE_TV || ri.resid;
      float acc = 0.0f;
      for (int base = v0 + threadIdx.x * 8; base < v1; base += kBatch * step) {
        float xt[kBatch][8], xd[kBatch][8];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          load8<DT>(j.T, (size_t)ri.trow * j.V, base + b * step, v1, vec, xt[b]);
          if (pair) load8<DT>(j.U, (size_t)ri.urow * j.V, base + b * step, v1, vec, xd[b]);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (base + b * step + i >= v1) continue;
            const float pt = prob_of(__fmul_rn(xt[b][i], j.scale), tn);
            if (!pair) {
              acc += pt;
              continue;
            }
            const float pd = draft_allowed(j, ri.r, base + b * step + i)
                                 ? prob_of(__fmul_rn(xd[b][i], j.scale), dn)
                                 : 0.0f;
            acc += MODE == MODE_RESID ? fmaxf(pt - pd, 0.0f) : fminf(pt, pd);
          }
        }
      }
      acc = block_sum(acc);
      if (threadIdx.x == 0) ps[out] = acc;
    }
  }
}

// Per-row softmax normaliser and/or argmax of target rows, one 512-thread block per row (two
// resident per SM): raw 16-byte words are loaded one batch ahead of the arithmetic, the maximum
// is tracked on the raw values (the scale is positive), exp((x - max) * scale) uses packed pair
// arithmetic, and (m, log Z) / the first argmax are written directly. Rows beyond a request's
// verified length are skipped.
constexpr int kRowThreads = 512;

__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long addx2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long mulx2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One 16-byte word (8 values) into the running (mx, s2, idx); s2 holds two partial sums.
template <int DT, bool STATS, bool ARGMAX>
__device__ __forceinline__ void row_word(const float (&x)[8], int v, float c, float& mx,
                                         unsigned long long& s2, int& idx) {
  const float g = fmaxf(fmax3(x[0], x[1], x[2]), fmax3(fmax3(x[3], x[4], x[5]), x[6], x[7]));
  if (g > mx) {
    if (ARGMAX) {
#pragma unroll
      for (int i = 7; i >= 0; --i)
        if (x[i] == g) idx = v + i;
    }
    if (STATS && mx > -INFINITY) {
      const float f = fast_exp2((mx - g) * c);
      s2 = mulx2(s2, pk2(f, f));
    }
    mx = g;
  }
  if (STATS && mx > -INFINITY) {  // words with no finite value so far add nothing (and no NaN)
    const unsigned long long nm = pk2(-mx, -mx), c2 = pk2(c, c);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      float a, b;
      upk2(mulx2(addx2(pk2(x[i], x[i + 1]), nm), c2), a, b);
      s2 = addx2(s2, pk2(fast_exp2(a), fast_exp2(b)));
    }
  }
}

// The normaliser part of row_word over a whole batch of words: one maximum and at most one
// rescale per batch instead of per word (fewer instructions per element; the same sum up to
// rounding).
template <int NB>
__device__ __forceinline__ void row_words_stats(const float (&x)[NB][8], float c, float& mx,
                                                unsigned long long& s2) {
  float g = mx;
#pragma unroll
  for (int b = 0; b < NB; ++b)
    g = fmaxf(g, fmaxf(fmax3(x[b][0], x[b][1], x[b][2]),
                       fmax3(fmax3(x[b][3], x[b][4], x[b][5]), x[b][6], x[b][7])));
  if (g > mx) {
    if (mx > -INFINITY) {
      const float f = fast_exp2((mx - g) * c);
      s2 = mulx2(s2, pk2(f, f));
    }
    mx = g;
  }
  if (mx > -INFINITY) {  // words with no finite value so far add nothing (and no NaN)
    const unsigned long long nm = pk2(-mx, -mx), c2 = pk2(c, c);
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        float a, bb;
        upk2(mulx2(addx2(pk2(x[b][i], x[b][i + 1]), nm), c2), a, bb);
        s2 = addx2(s2, pk2(fast_exp2(a), fast_exp2(bb)));
      }
  }
}

template <int DT>
__device__ __forceinline__ void unpack_word(const uint4& q, float (&x)[8]) {
  if constexpr (DT == SPEC_BF16) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

template <int DT, bool STATS, bool ARGMAX>
__global__ void __launch_bounds__(kRowThreads, 2) row_stats_kernel(RowJob j, bool vec, float* stats,
                                                                   int* argmax) {
  const int row = blockIdx.x;
  const RowInfo ri = row_info(j, row);
  if (!ri.active) return;
  const size_t off = (size_t)ri.trow * j.V;
  const float c = j.scale * kLog2e;
  float mx = -INFINITY;
  unsigned long long s2 = pk2(0.0f, 0.0f);
  int idx = 0x7fffffff;
  if (DT == SPEC_BF16 && vec) {
    // vector path: words w = tid + k * blockDim, kBatch words per batch, next batch in flight
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(j.T) + off);
    const int nw = j.V / 8;
    const int stride = kBatch * kRowThreads;
    uint4 cur[kBatch], nxt[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int w = threadIdx.x + b * kRowThreads;
      cur[b] = w < nw ? ld_stream16(p + w) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
    for (int w0 = threadIdx.x; w0 < nw; w0 += stride) {
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int w = w0 + stride + b * kRowThreads;
        nxt[b] = w < nw ? ld_stream16(p + w) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      }
      if constexpr (STATS && !ARGMAX) {
        float x[kBatch][8];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) unpack_word<DT>(cur[b], x[b]);  // padding: -inf
        row_words_stats<kBatch>(x, c, mx, s2);
      } else {
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          float x[8];
          unpack_word<DT>(cur[b], x);  // padding words decode to -inf
          row_word<DT, STATS, ARGMAX>(x, (w0 + b * kRowThreads) * 8, c, mx, s2, idx);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) cur[b] = nxt[b];
    }
  } else {
    for (int v = threadIdx.x * 8; v < j.V; v += kRowThreads * 8) {
      float x[8];
      load8<DT>(j.T, off, v, j.V, false, x);
      row_word<DT, STATS, ARGMAX>(x, v, c, mx, s2, idx);
    }
  }
  float sa, sb;
  upk2(s2, sa, sb);
  // merge in the scaled domain: (m = max * scale, s)
  StatsAcc a = {mx > -INFINITY ? __fmul_rn(mx, j.scale) : -INFINITY, sa + sb, idx};
  a = block_merge(a);
  if (threadIdx.x == 0) {
    if (STATS) {
      if (!(a.s > 0.0f) || !isfinite(a.s) || !(a.m > -INFINITY)) atomicOr(j.status, SPEC_DEV_NONFINITE);
      stats[2 * (size_t)row] = a.m;
      stats[2 * (size_t)row + 1] = logf(a.s);
    }
    if (ARGMAX) {
      int x = a.idx;
      if (x < 0 || x >= j.V) {
        atomicOr(j.status, SPEC_DEV_NONFINITE);
        x = 0;
      }
      argmax[row] = x;
    }
  }
}

// ------------------------------------------------------------------------------ generic Markov producer

// Softmax partials of Markov rows on CUDA cores with the W2 column tile staged once per block:
// a block takes a 64-column segment, copies its W2 rows into shared memory (coalesced, converted
// to fp32, rows padded by 16 bytes so that a row per thread reads without bank conflicts), then
// covers the rows four at a time: thread (row slot t / 64, column t % 64) runs the canonical fp32
// chain against the shared tile. The same arithmetic as draft_logit, so the partials are
// identical; only the memory traffic changes (each W2 row is read once per segment, not once per
// row). Needs rank <= 256, rank % 8 == 0 and 16-byte aligned weights.
constexpr int kTileCols = 64;
template <int UDT, int WDT, bool ARGMAX>
__global__ void __launch_bounds__(256) markov_ffma_tile(RowJob j, int nseg, float* pm, float* ps,
                                                        int* pi) {
  extern __shared__ __align__(16) float w2s[];  // [kTileCols][rank + 4]
  __shared__ __align__(16) float w1s[4][256];    // W1 rows of the four rows in flight
  __shared__ StatsAcc half[4][2];
  const int pitch = j.rank + 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = threadIdx.x >> 6, col = threadIdx.x & 63;
  const int k8 = j.rank / 8;  // 8-weight chunks per row
  for (int sg = blockIdx.x; sg < nseg; sg += gridDim.x) {
    const int v0 = sg * kTileCols;
    __syncthreads();  // the previous segment's tile is no longer read
    {
      // every chunk of this thread in flight before the first store
      constexpr int kIt = kTileCols * 32 / 256;  // chunks per thread at rank 256
      float x[kIt][8];
#pragma unroll
      for (int it = 0; it < kIt; ++it) {
        const int c = threadIdx.x + it * 256, rr = c / k8, q = c - rr * k8, v = v0 + rr;
#pragma unroll
        for (int t = 0; t < 8; ++t) x[it][t] = 0.0f;
        if (c < kTileCols * k8 && v < j.V) ld_w8<WDT>(j.W2, (size_t)v * j.rank + 8 * q, x[it]);
      }
#pragma unroll
      for (int it = 0; it < kIt; ++it) {
        const int c = threadIdx.x + it * 256, rr = c / k8, q = c - rr * k8;
        if (c < kTileCols * k8) {
          float4* d = reinterpret_cast<float4*>(w2s + rr * pitch + 8 * q);
          d[0] = make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
          d[1] = make_float4(x[it][4], x[it][5], x[it][6], x[it][7]);
        }
      }
    }
    __syncthreads();
    for (int r0 = 0; r0 < j.rows; r0 += 4) {
      const int row = r0 + slot, v = v0 + col;
      RowInfo ri;
      ri.prev = 0;
      if (row < j.rows) {
        ri = row_info(j, row);
        // the row's W1[prev] into shared memory: 64 threads, 8 weights each
        if (8 * col < j.rank) {
          float xa[8];
          ld_w8<WDT>(j.W1, (size_t)ri.prev * j.rank + 8 * col, xa);
          float4* d = reinterpret_cast<float4*>(&w1s[slot][8 * col]);
          d[0] = make_float4(xa[0], xa[1], xa[2], xa[3]);
          d[1] = make_float4(xa[4], xa[5], xa[6], xa[7]);
        }
      }
      __syncthreads();
      // columns past V take no part; a masked or non-finite column is a -inf entry
      StatsAcc e = stats_empty();
      if (row < j.rows && v < j.V) {
        e = {-INFINITY, 0.0f, v};
        if (draft_allowed(j, ri.r, v)) {
          float acc = 0.0f;
          const float* at = w1s[slot];
          const float* bt = w2s + col * pitch;
          for (int i0 = 0; i0 < j.rank; i0 += 8) {
            const float4 a0 = *reinterpret_cast<const float4*>(at + i0);
            const float4 a1 = *reinterpret_cast<const float4*>(at + i0 + 4);
            const float xa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float4 b0 = *reinterpret_cast<const float4*>(bt + i0);
            const float4 b1 = *reinterpret_cast<const float4*>(bt + i0 + 4);
            const float xb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int t = 0; t < 8; ++t) acc = __fmaf_rn(xa[t], xb[t], acc);
          }
          const float z = __fmul_rn(__fadd_rn(ld_elem<UDT>(j.U, (size_t)ri.urow * j.V + v), acc),
                                    j.scale);
          if (z > -INFINITY) e = {z, 1.0f, v};
        }
      }
      StatsAcc w = warp_merge(e);
      if (lane == 0) half[slot][warp & 1] = w;
      __syncthreads();
      if (col == 0 && row < j.rows) {
        const StatsAcc m = stats_merge(half[slot][0], half[slot][1]);
        const size_t out = (size_t)row * nseg + sg;
        pm[out] = m.m;
        ps[out] = m.s;
        if (ARGMAX) pi[out] = m.idx;
      }
      __syncthreads();
    }
  }
}


// One warp per (row, 64-column chunk); lane l handles columns c*64 + l and c*64 + 32 + l.
template <int UDT, int WDT, int MODE, bool ARGMAX>
__global__ void __launch_bounds__(256) markov_ffma_partials(RowJob j, int nseg, float* pm, float* ps,
                                                            int* pi) {
  const int lane = threadIdx.x & 31;
  const long long units = (long long)j.rows * nseg;
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long u = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
       u += stride) {
    const int row = (int)(u / nseg), c = (int)(u % nseg);
    const RowInfo ri = row_info(j, row);
    const size_t out = (size_t)row * nseg + c;
    if constexpr (MODE == MODE_STATS) {
      StatsAcc acc = stats_empty();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v = c * 64 + h * 32 + lane;
        if (v < j.V) {
          const float z = draft_logit<UDT, WDT>(j, ri, v);
          StatsAcc e = {z, 1.0f, v};
          if (!(z > -INFINITY)) e = {-INFINITY, 0.0f, v};
          acc = stats_merge(acc, e);
        }
      }
      acc = warp_merge(acc);
      if (lane == 0) {
        pm[out] = acc.m;
        ps[out] = acc.s;
        if (ARGMAX) pi[out] = acc.idx;
      }
    } else {
      Norm dn, tn;
      row_norms(j, ri, dn, tn);
      float acc = 0.0f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v = c * 64 + h * 32 + lane;
        if (v < j.V) acc += pair_value<UDT, WDT, MODE>(j, ri, dn, tn, v);
      }
      acc = warp_sum(acc);
      if (lane == 0) ps[out] = acc;
    }
  }
}

// ------------------------------------------------------------------------------ select

// One block per row: 256 threads, or 128 when the rows exceed one wave of 256-thread blocks
// (select.cuh has the select itself).
template <int UDT, int WDT>
__global__ void __launch_bounds__(256, 2) select_kernel(RowJob j, int seg, int nseg, const float* pm,
                                                     const float* ps, const int* pi,
                                                     SelectOut o) {
  __shared__ SelectShared sh;
  const int row = blockIdx.x;
  grid_dep_wait();  // the partials come from the kernel before
  if (row >= j.rows) return;
  const RowInfo ri = row_info(j, row);
  select_row<UDT, WDT, false>(j, ri, row, seg, nseg, pm, ps, pi, o, threadIdx.x, blockDim.x,
                              BlockBarrier{}, sh);
}


// ------------------------------------------------------------------------------ finalize / scans

// (m, log Z) per row from MODE_STATS partials; one warp per row.
__global__ void finalize_stats_kernel(int rows, int nseg, const float* pm, const float* ps,
                                      float* stats, const int32_t* lengths, int rows_per_req,
                                      uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  if (lengths && (row % rows_per_req) > min(max(lengths[row / rows_per_req], 0), rows_per_req - 1))
    return;  // row beyond the verified length: never read
  float M = -INFINITY;
  const float* rpm = pm + (size_t)row * nseg;
  const float* rps = ps + (size_t)row * nseg;
  for (int c = lane; c < nseg; c += 32) M = fmaxf(M, rpm[c]);
  M = warp_max(M);
  DF Z = df_zero();
  for (int c = lane; c < nseg; c += 32) {
    const float pmq = rpm[c], psq = rps[c];
    if (psq != 0.0f) Z = df_add(Z, psq * exp_shift(pmq, M));
  }
  Z = warp_sum_df(Z);
  if (lane == 0) {
    const bool zok = Z.hi > 0.0f && isfinite(Z.hi);
    if (!zok || !(M > -INFINITY)) atomicOr(status, SPEC_DEV_NONFINITE);
    stats[2 * (size_t)row] = M;
    stats[2 * (size_t)row + 1] = zok ? df_log(Z) : logf(Z.hi);
  }
}

// Greedy longest-prefix match + bonus, one thread per request, from per-row target argmaxes.
__global__ void greedy_scan_kernel(int R, int gamma, const int* amax, const int32_t* tokens,
                                   const int32_t* lengths, const int32_t* toff,
                                   int32_t* accept_len, int32_t* out_tokens,
                                   int32_t* next_anchor, uint32_t* status) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  int l = gamma;
  if (lengths) {
    l = lengths[r];
    if (l < 0 || l > gamma) {
      atomicOr(status, SPEC_DEV_BAD_LENGTH);
      l = l < 0 ? 0 : gamma;
    }
  }
  int n = 0, y = 0;
  for (int i = 0; i <= l; ++i) {
    y = amax[target_row(toff, R, gamma, r, i, status)];
    if (i == l || tokens[(size_t)r * gamma + i] != y) break;
    n = i + 1;
  }
  accept_len[r] = n;
  if (out_tokens) {
    int32_t* o = out_tokens + (size_t)r * (gamma + 1);
    for (int i = 0; i <= gamma; ++i) o[i] = i < n ? tokens[(size_t)r * gamma + i] : -1;
    o[n] = y;
  }
  if (next_anchor) next_anchor[r] = y;
}

// Rejection-sampling acceptance scan, one warp per request: lane k tests position k+1
// (accept x_k iff u_accept * p_d(x_k) < p_t,k-1(x_k); the tests are independent), and n_r is
// the first failing position. Records n_r and whether the final token is a residual draw
// (a rejection) or a bonus draw (all l accepted).
template <int DT>
__global__ void accept_kernel(int R, int gamma, int V, float scale, const void* T,
                              const float* tstats, const int32_t* tokens, const float* dlogp,
                              const float* u_accept, const int32_t* lengths,
                              const int32_t* toff, int32_t* final_n, int32_t* final_kind,
                              int32_t* accept_len, int32_t* out_tokens, uint32_t* status,
                              RowPrefetch pf) {
  grid_dep_wait();  // the target normalisers may come from the kernel before
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= R) return;
  int l = gamma;
  if (lengths) {
    l = lengths[r];
    if (l < 0 || l > gamma) {
      if (lane == 0) atomicOr(status, SPEC_DEV_BAD_LENGTH);
      l = l < 0 ? 0 : gamma;
    }
  }
  int n = l;
  for (int k0 = 0; k0 < l && n == l; k0 += 32) {
    const int k = k0 + lane;  // tests position k + 1
    bool reject = false;
    if (k < l) {
      const int x = tokens[(size_t)r * gamma + k];
      if (x < 0 || x >= V) {
        atomicOr(status, SPEC_DEV_BAD_TOKEN);
        reject = true;  // an invalid proposal is rejected
      } else {
        const long long trow = target_row(toff, R, gamma, r, k, status);
        const float t = __fmul_rn(ld_elem<DT>(T, (size_t)trow * V + x), scale);
        const float pt = prob_of(t, load_norm(tstats, trow));
        const float pd = fast_exp2(dlogp[(size_t)r * gamma + k] * kLog2e);  // exp(log p_d)
        reject = !(u_accept[(size_t)r * gamma + k] * pd < pt);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, reject);
    if (m) n = k0 + __ffs(m) - 1;
  }
  if (lane == 0) {
    final_n[r] = n;
    final_kind[r] = n < l ? 1 : 0;
    accept_len[r] = n;
    if (pf.w1) {  // the residual pass gathers W1 of the final row's previous token
      const int prev = n == 0 ? pf.anchors[r] : tokens[(size_t)r * gamma + n - 1];
      if (prev >= 0 && prev < V)
        l2_prefetch_bytes(static_cast<const char*>(pf.w1) + (size_t)prev * pf.row_bytes,
                          pf.row_bytes);
    }
  }
  if (out_tokens) {
    int32_t* o = out_tokens + (size_t)r * (gamma + 1);
    for (int i = lane; i <= gamma; i += 32) o[i] = i < n ? tokens[(size_t)r * gamma + i] : -1;
  }
}

// c*_{r,k} = sum of the MODE_TV partials of row (r, k), clamped to [0, 1]; survival
// a_{r,j} = fl32(a_{r,j-1} * c_{r,j}) in order. One warp per request.
__global__ void tv_finalize_kernel(int R, int gamma, int nseg, const float* ps, float* conf,
                                   float* survival) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= R) return;
  float a = 1.0f;
  for (int k = 0; k < gamma; ++k) {
    const int row = r * gamma + k;
    DF c = df_zero();
    for (int s = lane; s < nseg; s += 32) c = df_add(c, ps[(size_t)row * nseg + s]);
    c = warp_sum_df(c);
    if (lane == 0) {
      float cf = df_float(c);
      cf = fminf(fmaxf(cf, 0.0f), 1.0f);
      a = __fmul_rn(a, cf);
      conf[row] = cf;
      if (survival) survival[row] = a;
    }
  }
}

// ------------------------------------------------------------------------------ launchers

namespace {
template <int DT, int MODE, bool SUM, bool ARGMAX>
void launch_stream_t(const RowJob& j, int seg, int nseg, bool vec, float* pm, float* ps, int* pi,
                     int grid, cudaStream_t s) {
  stream_partials_kernel<DT, MODE, SUM, ARGMAX><<<grid, 256, 0, s>>>(j, seg, nseg, vec, pm, ps, pi);
}

template <int UDT, int WDT>
void launch_ffma_t(const RowJob& j, int nseg, bool argmax, float* pm, float* ps, int* pi, int grid,
                   cudaStream_t s) {
  const bool tile = j.mode == MODE_STATS && j.rank > 0 && j.rank <= 256 && j.rank % 8 == 0 &&
                    ((reinterpret_cast<uintptr_t>(j.W1) | reinterpret_cast<uintptr_t>(j.W2)) & 15) == 0;
  if (tile) {
    const size_t smem = (size_t)kTileCols * (j.rank + 4) * sizeof(float);
    const int g = nseg < num_sms() * 3 ? nseg : num_sms() * 3;
    if (argmax) {
      cudaFuncSetAttribute(markov_ffma_tile<UDT, WDT, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      markov_ffma_tile<UDT, WDT, true><<<g, 256, smem, s>>>(j, nseg, pm, ps, pi);
    } else {
      cudaFuncSetAttribute(markov_ffma_tile<UDT, WDT, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      markov_ffma_tile<UDT, WDT, false><<<g, 256, smem, s>>>(j, nseg, pm, ps, pi);
    }
    return;
  }
  switch (j.mode) {
    case MODE_STATS:
      if (argmax)
        markov_ffma_partials<UDT, WDT, MODE_STATS, true><<<grid, 256, 0, s>>>(j, nseg, pm, ps, pi);
      else
        markov_ffma_partials<UDT, WDT, MODE_STATS, false><<<grid, 256, 0, s>>>(j, nseg, pm, ps, pi);
      break;
    case MODE_RESID:
      markov_ffma_partials<UDT, WDT, MODE_RESID, false><<<grid, 256, 0, s>>>(j, nseg, pm, ps, pi);
      break;
    default:
      markov_ffma_partials<UDT, WDT, MODE_TV, false><<<grid, 256, 0, s>>>(j, nseg, pm, ps, pi);
      break;
  }
}
}  // namespace

void launch_row_stats(const RowJob& j, int dtype, bool vec, float* stats, int* argmax,
                      cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_STREAM, s);
  if (j.rows == 0) return;
  const bool st = stats != nullptr, am = argmax != nullptr;
  if (dtype == SPEC_BF16) {
    if (st && am) row_stats_kernel<SPEC_BF16, true, true><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
    else if (st) row_stats_kernel<SPEC_BF16, true, false><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
    else row_stats_kernel<SPEC_BF16, false, true><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
  } else {
    if (st && am) row_stats_kernel<SPEC_F32, true, true><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
    else if (st) row_stats_kernel<SPEC_F32, true, false><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
    else row_stats_kernel<SPEC_F32, false, true><<<j.rows, kRowThreads, 0, s>>>(j, vec, stats, argmax);
  }
}

void launch_stream_partials(const RowJob& j, int dtype, int seg, int nseg, bool vec, bool sum,
                            bool argmax, float* pm, float* ps, int* pi, int grid, cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_STREAM, s);
  if (dtype == SPEC_BF16) {
    switch (j.mode) {
      case MODE_STATS:
        if (sum && argmax) launch_stream_t<SPEC_BF16, MODE_STATS, true, true>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        else if (sum) launch_stream_t<SPEC_BF16, MODE_STATS, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        else launch_stream_t<SPEC_BF16, MODE_STATS, false, true>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        break;
      case MODE_RESID: launch_stream_t<SPEC_BF16, MODE_RESID, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s); break;
      default: launch_stream_t<SPEC_BF16, MODE_TV, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s); break;
    }
  } else {
    switch (j.mode) {
      case MODE_STATS:
        if (sum && argmax) launch_stream_t<SPEC_F32, MODE_STATS, true, true>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        else if (sum) launch_stream_t<SPEC_F32, MODE_STATS, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        else launch_stream_t<SPEC_F32, MODE_STATS, false, true>(j, seg, nseg, vec, pm, ps, pi, grid, s);
        break;
      case MODE_RESID: launch_stream_t<SPEC_F32, MODE_RESID, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s); break;
      default: launch_stream_t<SPEC_F32, MODE_TV, true, false>(j, seg, nseg, vec, pm, ps, pi, grid, s); break;
    }
  }
}

void launch_ffma_partials(const RowJob& j, int udt, int wdt, int nseg, bool argmax, float* pm,
                          float* ps, int* pi, int grid, cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_MARKOV, s);
  if (udt == SPEC_BF16 && wdt == SPEC_BF16) launch_ffma_t<SPEC_BF16, SPEC_BF16>(j, nseg, argmax, pm, ps, pi, grid, s);
  else if (udt == SPEC_BF16) launch_ffma_t<SPEC_BF16, SPEC_F32>(j, nseg, argmax, pm, ps, pi, grid, s);
  else if (wdt == SPEC_BF16) launch_ffma_t<SPEC_F32, SPEC_BF16>(j, nseg, argmax, pm, ps, pi, grid, s);
  else launch_ffma_t<SPEC_F32, SPEC_F32>(j, nseg, argmax, pm, ps, pi, grid, s);
}

void launch_select(const RowJob& j, int udt, int wdt, int seg, int nseg, const float* pm,
                   const float* ps, const int* pi, const SelectOut& o, cudaStream_t s) {
  if (j.rows == 0) return;
  TraceScope ts(SPEC_KCLASS_SELECT, s);
  // two 256-thread blocks fit an SM; beyond one wave of those, 128-thread blocks (four per SM)
  // halve the number of waves at some cost per row
  const int nt = j.rows > 2 * num_sms() ? 128 : 256;
  auto k = udt == SPEC_BF16 ? (wdt == SPEC_BF16 ? select_kernel<SPEC_BF16, SPEC_BF16>
                                                : select_kernel<SPEC_BF16, SPEC_F32>)
                            : (wdt == SPEC_BF16 ? select_kernel<SPEC_F32, SPEC_BF16>
                                                : select_kernel<SPEC_F32, SPEC_F32>);
  launch_kernel(k, dim3(j.rows), dim3(nt), 0, s, j.pdl != 0, j, seg, nseg, pm, ps, pi, o);
}

void launch_finalize_stats(int rows, int nseg, const float* pm, const float* ps, float* stats,
                           const int32_t* lengths, int rows_per_req, uint32_t* status,
                           cudaStream_t s) {
  if (rows == 0) return;
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  finalize_stats_kernel<<<(rows + 7) / 8, 256, 0, s>>>(rows, nseg, pm, ps, stats, lengths,
                                                        rows_per_req, status);
}

void launch_greedy_scan(int R, int gamma, const int* amax, const int32_t* tokens,
                        const int32_t* lengths, const int32_t* toff, int32_t* accept_len,
                        int32_t* out_tokens, int32_t* next_anchor, uint32_t* status,
                        cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  greedy_scan_kernel<<<(R + 127) / 128, 128, 0, s>>>(R, gamma, amax, tokens, lengths, toff,
                                                     accept_len, out_tokens, next_anchor, status);
}

void launch_accept(int dtype, int R, int gamma, int V, float scale, const void* T,
                   const float* tstats, const int32_t* tokens, const float* dlogp,
                   const float* u_accept, const int32_t* lengths, const int32_t* toff,
                   int32_t* final_n, int32_t* final_kind, int32_t* accept_len,
                   int32_t* out_tokens, uint32_t* status, RowPrefetch pf, bool chained,
                   cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  const int grid = (R + 7) / 8;  // one warp per request, 8 warps per block
  launch_kernel(dtype == SPEC_BF16 ? accept_kernel<SPEC_BF16> : accept_kernel<SPEC_F32>,
                dim3(grid), dim3(256), 0, s, chained, R, gamma, V, scale, T, tstats, tokens,
                dlogp, u_accept, lengths, toff, final_n, final_kind, accept_len, out_tokens,
                status, pf);
}

void launch_tv_finalize(int R, int gamma, int nseg, const float* ps, float* conf, float* survival,
                        cudaStream_t s) {
  TraceScope ts(SPEC_KCLASS_OTHER, s);
  tv_finalize_kernel<<<(R + 7) / 8, 256, 0, s>>>(R, gamma, nseg, ps, conf, survival);
}

}  // namespace spec
