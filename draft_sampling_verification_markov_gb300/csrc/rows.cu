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

namespace spec {

// ------------------------------------------------------------------------------ logits

// 8 consecutive weights from a 16-byte aligned address, as fp32.
template <int WDT>
__device__ __forceinline__ void ld_w8(const void* p, size_t i, float* x) {
  if constexpr (WDT == SPEC_BF16) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p) + i));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      x[2 * t] = __uint_as_float(w[t] << 16);
      x[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
  } else {
    const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
    const float4 a = __ldg(f), b = __ldg(f + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Markov bias W1[prev] . W2[v] in the canonical fp32 chain acc = fma(W1[prev][i], W2[v][i], acc),
// i ascending. With 16-byte aligned rows the weights come 8 at a time, 32 in flight, and the
// chain is unchanged, so the result is bit-identical to the element-by-element loop.
template <int WDT>
__device__ __forceinline__ float markov_bias(const RowJob& j, int prev, int v) {
  float acc = 0.0f;
  const size_t a = (size_t)prev * j.rank, b = (size_t)v * j.rank;
  const bool vec = (j.rank & 7) == 0 &&
                   ((reinterpret_cast<uintptr_t>(j.W1) | reinterpret_cast<uintptr_t>(j.W2)) & 15) == 0;
  if (vec) {
    constexpr int kChunk = 32;  // weights in flight per operand (registers are scarce in select)
    for (int i0 = 0; i0 < j.rank; i0 += kChunk) {
      float xa[kChunk], xb[kChunk];
#pragma unroll
      for (int t = 0; t < kChunk / 8; ++t)
        if (i0 + 8 * t < j.rank) {
          ld_w8<WDT>(j.W1, a + i0 + 8 * t, xa + 8 * t);
          ld_w8<WDT>(j.W2, b + i0 + 8 * t, xb + 8 * t);
        }
#pragma unroll
      for (int t = 0; t < kChunk; ++t)
        if (i0 + t < j.rank) acc = __fmaf_rn(xa[t], xb[t], acc);
    }
  } else {
    for (int i = 0; i < j.rank; ++i)
      acc = __fmaf_rn(ld_elem<WDT>(j.W1, a + i), ld_elem<WDT>(j.W2, b + i), acc);
  }
  return acc;
}

// Draft logit z_d(v) of a row (DSpark sections 3-4): (U + W1[prev] . W2[v]) * scale, the bias
// in the canonical fp32 chain.
template <int UDT, int WDT>
__device__ __forceinline__ float draft_logit(const RowJob& j, const RowInfo& ri, int v) {
  if (!draft_allowed(j, ri.r, v)) return -INFINITY;
  const float acc = j.rank > 0 ? markov_bias<WDT>(j, ri.prev, v) : 0.0f;
  const float s = __fadd_rn(ld_elem<UDT>(j.U, (size_t)ri.urow * j.V + v), acc);
  return __fmul_rn(s, j.scale);
}

template <int DT>
__device__ __forceinline__ float target_logit(const RowJob& j, const RowInfo& ri, int v) {
  return __fmul_rn(ld_elem<DT>(j.T, (size_t)ri.trow * j.V + v), j.scale);
}

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

// Exclusive block scan of one double-float per thread; returns the exclusive prefix and writes
// the block total.
__device__ __forceinline__ DF block_exscan_df(DF x, DF* total) {
  __shared__ DF sm[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const DF inc = warp_scan_df(x);
  DF ex = df_shfl_up(inc, 1);
  if (lane == 0) ex = df_zero();
  __syncthreads();
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const DF w = lane < nw ? sm[lane] : df_zero();
    const DF wi = warp_scan_df(w);
    DF wex = df_shfl_up(wi, 1);
    if (lane == 0) wex = df_zero();
    if (lane < nw) sm[lane] = wex;
    if (lane == nw - 1) sm[32] = wi;
  }
  __syncthreads();
  const DF r = df_add(sm[warp], ex);
  *total = sm[32];
  __syncthreads();
  return r;
}

// Value of element v of the crossing segment: exp(z_d - M) for a proposal, or the residual /
// bonus mass q(v) for a final draw; z_d is passed in (bias already included).
template <int UDT, int WDT>
__device__ __forceinline__ float seg_value(const RowJob& j, const RowInfo& ri, bool resid,
                                           float M, Norm dn, Norm tn, int v, float zd) {
  if (!resid) return exp_shift(zd, M);
  const float pt = prob_of(target_logit<UDT>(j, ri, v), tn);
  if (!ri.resid) return pt;
  return fmaxf(pt - prob_of(zd, dn), 0.0f);
}

// Draft logits of columns [v0, v0 + n) (n <= 64) into zs[], using all 256 threads. bf16
// weights: a split-K dot product (256/64.. threads per column, 16-byte loads, shuffle
// reduction); fp32 weights: the canonical fp32 chain, one thread per column.
template <int UDT, int WDT>
__device__ void segment_logits(const RowJob& j, const RowInfo& ri, int v0, int n, float* zs) {
  const int tid = threadIdx.x;
  if (WDT == SPEC_BF16 && j.rank > 0 && (j.rank % 8) == 0) {
    const int tpc = blockDim.x / 64;          // threads per column (4)
    const int col = tid / tpc, part = tid % tpc;
    const int v = v0 + col;
    float acc = 0.0f;
    // the base logit is independent of the dot product: its load goes out first
    const float uval = col < n && part == 0 ? ld_elem<UDT>(j.U, (size_t)ri.urow * j.V + v) : 0.0f;
    if (col < n) {
      const uint4* w1 = reinterpret_cast<const uint4*>(
          reinterpret_cast<const unsigned short*>(j.W1) + (size_t)ri.prev * j.rank);
      const uint4* w2 = reinterpret_cast<const uint4*>(
          reinterpret_cast<const unsigned short*>(j.W2) + (size_t)v * j.rank);
      const int nc = j.rank / 8;  // 16-byte chunks per weight row
      for (int c0 = part; c0 < nc; c0 += 8 * tpc) {
        // up to 8 chunk pairs per thread in flight before any arithmetic
        uint4 a[8], b[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = c0 + q * tpc;
          a[q] = c < nc ? __ldg(w1 + c) : make_uint4(0, 0, 0, 0);
          b[q] = c < nc ? __ldg(w2 + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t aa[4] = {a[q].x, a[q].y, a[q].z, a[q].w};
          const uint32_t bb[4] = {b[q].x, b[q].y, b[q].z, b[q].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(aa[e] << 16), __uint_as_float(bb[e] << 16), acc);
            acc = fmaf(__uint_as_float(aa[e] & 0xffff0000u), __uint_as_float(bb[e] & 0xffff0000u),
                       acc);
          }
        }
      }
    }
    for (int off = tpc / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (col < n && part == 0) {
      const float s = __fadd_rn(uval, acc);
      zs[col] = draft_allowed(j, ri.r, v) ? __fmul_rn(s, j.scale) : -INFINITY;
    }
  } else {
    if (tid < n) zs[tid] = draft_logit<UDT, WDT>(j, ri, v0 + tid);
  }
  __syncthreads();
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void l2_prefetch_bytes(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One block per row: 256 threads, or 128 when the rows exceed one wave of 256-thread blocks.
//   kind 0 (MODE_STATS partials): greedy argmax, or inverse-CDF draw from the softmax;
//   kind 1 (MODE_RESID partials): inverse-CDF draw from the residual / bonus distribution.
// Only the crossing segment is recomputed element by element; everything else uses the
// partials. Markov segments (<= 64 columns) are rebuilt once into shared memory.
template <int UDT, int WDT>
__global__ void __launch_bounds__(256, 2) select_kernel(RowJob j, int seg, int nseg, const float* pm,
                                                     const float* ps, const int* pi,
                                                     SelectOut o) {
  __shared__ int sh_c, sh_x, sh_last;
  __shared__ float sh_rem;
  __shared__ float sh_M, sh_lz;
  __shared__ float zs[64];   // draft logits of the segment starting at sh_zv0
  __shared__ float es[64];
  __shared__ int sh_zv0;
  const int row = blockIdx.x;
  grid_dep_wait();  // the partials come from the kernel before
  if (row >= j.rows) return;
  const RowInfo ri = row_info(j, row);
  const int tid = threadIdx.x;
  const bool resid = o.kind == 1;
  const float u_row = (o.greedy && !resid) ? 0.0f : o.uni[(size_t)row * o.uni_stride + o.uni_offset];
  const bool markov = resid ? (ri.resid && j.rank > 0) : j.rank > 0;
  const bool need_z = j.rank > 0 && (!resid || ri.resid);

  // 1. normaliser from the partials. Warp w owns the contiguous segment range [s0, s1) of the
  // row's (row-major) partials and lane l a contiguous run [c0, c1) of it; a run of up to kPer
  // segments stays in registers through the crossing search below.
  const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int s0 = (int)((long long)nseg * warp / nwarps);
  const int s1 = (int)((long long)nseg * (warp + 1) / nwarps);
  const int per = (s1 - s0 + 31) / 32;
  const int c0 = min(s1, s0 + lane * per), c1 = min(s1, c0 + per);
  const float* rpm = pm + (size_t)row * nseg;
  const float* rps = ps + (size_t)row * nseg;
  constexpr int kPer = 16;
  const bool in_regs = per <= kPer;  // the same for every thread of the block
  float lm[kPer], ls[kPer];
  float M = -INFINITY;
  int gidx = 0x7fffffff;
  if (!resid) {
    // only the row maximum and its first index are needed here (Z comes from the weights
    // below): a max / min-index reduction, no exponentials
    const int* rpi = pi ? pi + (size_t)row * nseg : nullptr;
    float lmax = -INFINITY;
    int lidx = 0x7fffffff;
    if (in_regs) {
      int li[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int c = c0 + k;
        lm[k] = -INFINITY;
        ls[k] = 0.0f;
        li[k] = 0x7fffffff;
        if (c < c1) {
          lm[k] = rpm[c];
          ls[k] = rps[c];
          if (rpi) li[k] = rpi[c];
        }
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) lmax = fmaxf(lmax, lm[k]);
      if (rpi) {
#pragma unroll
        for (int k = 0; k < kPer; ++k)
          if (lm[k] == lmax && li[k] < lidx) lidx = li[k];
      }
    } else {
      for (int c = c0; c < c1; ++c) {
        const float v = rpm[c];
        const int ix = rpi ? rpi[c] : 0x7fffffff;
        if (v > lmax || (v == lmax && ix < lidx)) {
          lmax = v;
          lidx = ix;
        }
      }
    }
    // warp, then block: larger maximum wins, equal maxima keep the lower index
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, lmax, off);
      const int oi = __shfl_xor_sync(0xffffffffu, lidx, off);
      if (om > lmax || (om == lmax && oi < lidx)) {
        lmax = om;
        lidx = oi;
      }
    }
    __shared__ float sh_wm[32];
    __shared__ int sh_wi[32];
    if (lane == 0) {
      sh_wm[warp] = lmax;
      sh_wi[warp] = lidx;
    }
    __syncthreads();
    for (int w = 0; w < nwarps; ++w) {
      const float om = sh_wm[w];
      const int oi = sh_wi[w];
      if (om > M || (om == M && oi < gidx)) {
        M = om;
        gidx = oi;
      }
    }
  }
  // 2. segment weights (each partial's share of Z, fp32); run sums, an inclusive warp scan of
  // them and the warp totals as double-float pairs; Z and every warp's offset are sums of the
  // warp totals in warp order
  auto weight = [&](float pmv, float psv) -> float {
    return resid ? psv : (psv == 0.0f ? 0.0f : psv * exp_shift(pmv, M));
  };
  DF lsum = df_zero();
  if (in_regs) {
    if (resid) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        lm[k] = 0.0f;
        ls[k] = c0 + k < c1 ? rps[c0 + k] : 0.0f;
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      ls[k] = c0 + k < c1 ? weight(lm[k], ls[k]) : 0.0f;  // ls now holds the weights
      lsum = df_add(lsum, ls[k]);
    }
  } else {
    for (int c = c0; c < c1; ++c) lsum = df_add(lsum, weight(resid ? 0.0f : rpm[c], rps[c]));
  }
  const DF incl = warp_scan_df(lsum);
  DF run_before = df_shfl_up(incl, 1);  // the warp's mass before this run
  if (lane == 0) run_before = df_zero();
  __shared__ DF sh_wt[32];
  if (lane == 31) sh_wt[warp] = incl;
  __syncthreads();
  DF Z = df_zero();
  for (int w = 0; w < nwarps; ++w) Z = df_add(Z, sh_wt[w]);
  if (tid == 0) {
    sh_M = M;
    const bool zok = Z.hi > 0.0f && isfinite(Z.hi);
    sh_lz = resid ? 0.0f : (zok ? df_log(Z) : logf(Z.hi));
    sh_c = -1;
    sh_rem = 0.0f;
    sh_x = -1;
    sh_last = -1;
    sh_zv0 = -1;
    if (!resid && (!zok || !(M > -INFINITY))) atomicOr(j.status, SPEC_DEV_NONFINITE);
  }
  __syncthreads();

  int x = -1;
  if (!resid && o.greedy) {
    x = gidx;
    if (x < 0 || x >= j.V) {
      if (tid == 0) atomicOr(j.status, SPEC_DEV_NONFINITE);
      x = 0;
    }
    if (markov && o.logp) {  // rebuild the segment holding x for its log-probability
      const int v0 = (x / 64) * 64;
      segment_logits<UDT, WDT>(j, ri, v0, min(64, j.V - v0), zs);
      if (tid == 0) sh_zv0 = v0;
      __syncthreads();
    }
  } else {
    // 3. crossing segment for t = u * Z: the warp whose mass holds t, the first lane of it
    // whose cumulative mass exceeds t, then that lane's run in order
    const DF t = df_mul(Z, u_row);
    DF before = df_zero();
    int wstar = -1;
    for (int w = 0; w < nwarps; ++w) {
      const DF next = df_add(before, sh_wt[w]);
      if (df_gt(next, t)) {
        wstar = w;
        break;
      }
      before = next;
    }
    if (warp == wstar) {
      const unsigned hit = __ballot_sync(0xffffffffu, df_gt(df_add(before, incl), t));
      if (hit && lane == __ffs(hit) - 1) {
        DF cum = df_add(before, run_before);
        int found = -1, lastpos = -1;
        float remv = 1e30f;
        if (in_regs) {
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            if (found < 0 && c0 + k < c1) {
              const float wv = ls[k];
              const DF next = df_add(cum, wv);
              if (df_gt(next, t)) {
                found = c0 + k;
                remv = df_float(df_add(t, df_neg(cum)));
              }
              if (wv > 0.0f) lastpos = c0 + k;
              cum = next;
            }
          }
        } else {
          for (int c = c0; c < c1 && found < 0; ++c) {
            const float wv = weight(resid ? 0.0f : rpm[c], rps[c]);
            const DF next = df_add(cum, wv);
            if (df_gt(next, t)) {
              found = c;
              remv = df_float(df_add(t, df_neg(cum)));
            }
            if (wv > 0.0f) lastpos = c;
            cum = next;
          }
        }
        // without a crossing in the run (summation-order rounding) the draw ends the run's
        // last segment with positive mass
        sh_c = found >= 0 ? found : lastpos;
        sh_rem = found >= 0 ? remv : 1e30f;
      }
    }
    __syncthreads();
    if (sh_c < 0 && tid == 0) {
      // rounding left no crossing: the end of the last segment with positive mass
      int last = -1;
      for (int c = nseg - 1; c >= 0 && last < 0; --c)
        if (rps[c] > 0.0f) last = c;
      if (last < 0) atomicOr(j.status, resid ? SPEC_DEV_EMPTY_RESIDUAL : SPEC_DEV_NONFINITE);
      sh_c = last;
      sh_rem = 1e30f;
    }
    __syncthreads();
    const int cstar = sh_c;
    const float rem = sh_rem;
    Norm dn = {0.0f, 0.0f}, tn = {0.0f, 0.0f};
    if (resid) row_norms(j, ri, dn, tn);
    const int v0 = max(cstar, 0) * seg, v1 = min(j.V, v0 + seg);
    if (seg <= 64) {
      // 3a. small segment: values into shared memory, warp 0 scans in token order
      if (need_z) {
        segment_logits<UDT, WDT>(j, ri, v0, v1 - v0, zs);
        if (tid == 0) sh_zv0 = v0;
      }
      for (int e = tid; e < v1 - v0; e += blockDim.x) {
        const float zd = need_z ? zs[e] : (ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v0 + e) : 0.0f);
        es[e] = seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v0 + e, zd);
      }
      __syncthreads();
      if (tid < 32 && cstar >= 0) {
        const int n = v1 - v0;
        float a0 = tid < n ? es[tid] : 0.0f, a1 = tid + 32 < n ? es[tid + 32] : 0.0f;
        float s0 = a0, s1 = a1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y0 = __shfl_up_sync(0xffffffffu, s0, off);
          const float y1 = __shfl_up_sync(0xffffffffu, s1, off);
          if (tid >= off) {
            s0 += y0;
            s1 += y1;
          }
        }
        const float tot0 = __shfl_sync(0xffffffffu, s0, 31);
        s1 += tot0;
        const unsigned m0 = __ballot_sync(0xffffffffu, s0 > rem && tid < n);
        const unsigned m1 = __ballot_sync(0xffffffffu, s1 > rem && tid + 32 < n);
        const unsigned p0 = __ballot_sync(0xffffffffu, a0 > 0.0f), p1 = __ballot_sync(0xffffffffu, a1 > 0.0f);
        if (tid == 0) {
          if (m0) sh_x = v0 + __ffs(m0) - 1;
          else if (m1) sh_x = v0 + 32 + __ffs(m1) - 1;
          sh_last = p1 ? v0 + 32 + 31 - __clz(p1) : (p0 ? v0 + 31 - __clz(p0) : -1);
        }
      }
    } else {
      // 3b. long segment (no Markov bias): per-thread runs, block scan, rescan one run
      const int per = (seg + blockDim.x - 1) / blockDim.x;
      const int e0 = min(v1, v0 + tid * per), e1 = min(v1, e0 + per);
      DF mine = df_zero();
      for (int v = e0; v < e1; ++v)
        mine = df_add(mine, seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                                ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f));
      DF segtot;
      const DF sbefore = block_exscan_df(mine, &segtot);
      const DF r = {rem, 0.0f};
      if (cstar >= 0) {
        if (!df_gt(sbefore, r) && df_gt(df_add(sbefore, mine), r)) {
          DF cum = sbefore;
          for (int v = e0; v < e1; ++v) {
            const float w = seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                                ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f);
            cum = df_add(cum, w);
            if (df_gt(cum, r)) {
              sh_x = v;
              break;
            }
          }
        }
        int lastp = -1;
        for (int v = e1 - 1; v >= e0 && lastp < 0; --v)
          if (seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                  ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f) > 0.0f)
            lastp = v;
        if (lastp >= 0) atomicMax(&sh_last, lastp);
      }
    }
    __syncthreads();
    x = sh_x >= 0 ? sh_x : sh_last;
    if (x < 0) {
      // no mass at all: emit a valid id (the proposed token at the rejected position for a
      // residual, token 0 otherwise); the status word already records the fault
      x = 0;
      if (resid && ri.resid) {
        const int n = j.final_n[row];
        x = j.tokens[(size_t)row * j.gamma + n];
        if (x < 0 || x >= j.V) x = 0;
      }
    }
  }

  // 4. outputs
  if (tid == 0) {
    if (!resid) {
      // the row's (request, position): one position per pass, or all of them (no Markov head)
      const size_t q = j.map == MAP_ALL_POS ? (size_t)row : (size_t)row * j.gamma + (j.k - 1);
      o.tokens[q] = x;
      if (o.w1) l2_prefetch_bytes(static_cast<const char*>(o.w1) + (size_t)x * o.w1_row_bytes,
                                  o.w1_row_bytes);
      if (o.logp) {
        const int zv0 = sh_zv0;
        const float zx = (zv0 >= 0 && x >= zv0 && x < zv0 + 64) ? zs[x - zv0]
                                                                : draft_logit<UDT, WDT>(j, ri, x);
        o.logp[q] = zx - sh_M - sh_lz;
      }
      if (o.stats) {
        o.stats[2 * q] = sh_M;
        o.stats[2 * q + 1] = sh_lz;
      }
    } else {
      const int n = j.final_n[row];
      o.tokens[(size_t)row * (j.gamma + 1) + n] = x;
      if (o.next_anchor) o.next_anchor[row] = x;
      if (o.w1) l2_prefetch_bytes(static_cast<const char*>(o.w1) + (size_t)x * o.w1_row_bytes,
                                  o.w1_row_bytes);
    }
  }
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
