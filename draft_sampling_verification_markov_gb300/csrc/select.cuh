// select.cuh -- the per-row select of libspecmarkov, shared by the select kernel (one block
// per row) and the persistent proposal kernel (one warpgroup per row).
//
// A select combines the partials a producer wrote for one row: the row maximum and normaliser
// from the per-segment (max, sum exp) pairs, then the greedy argmax or the inverse-CDF draw of
// the caller's uniform ("[DeepSeek-6] DSpark", section 3: softmax of U_k + B_k and sampling;
// section 4: the Markov bias). Only the segment in which the cumulative mass crosses u * Z is
// rebuilt element by element.
#pragma once

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

// ------------------------------------------------------------------------------ select

// Barrier over the threads that run one select: the whole block, or a named barrier of a
// warpgroup inside a larger block.
struct BlockBarrier {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
struct NamedBarrier {
  int id, count;
  __device__ __forceinline__ void operator()() const {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
  }
};

// Partials are read through L2 (not L1) when other CTAs of the same launch write them.
template <bool COHERENT, typename T>
__device__ __forceinline__ T ld_part(const T* p) {
  if constexpr (COHERENT) return __ldcg(p);
  else return *p;
}

// Shared state of one select.
struct SelectShared {
  int c, x, last, zv0;
  float rem, M, lz;
  float zs[64];  // draft logits of the segment starting at zv0
  float es[64];
  float wm[32];
  int wi[32];
  DF wt[32];
  DF scan[33];
};

// Exclusive scan of one double-float per thread over the select's threads; returns the
// exclusive prefix and writes the total.
template <class Sync>
__device__ __forceinline__ DF block_exscan_df(DF x, DF* total, int tid, int nthreads, Sync sync,
                                              DF* sm) {
  const int lane = tid & 31, warp = tid >> 5, nw = nthreads >> 5;
  const DF inc = warp_scan_df(x);
  DF ex = df_shfl_up(inc, 1);
  if (lane == 0) ex = df_zero();
  sync();
  if (lane == 31) sm[warp] = inc;
  sync();
  if (warp == 0) {
    const DF w = lane < nw ? sm[lane] : df_zero();
    const DF wi = warp_scan_df(w);
    DF wex = df_shfl_up(wi, 1);
    if (lane == 0) wex = df_zero();
    if (lane < nw) sm[lane] = wex;
    if (lane == nw - 1) sm[32] = wi;
  }
  sync();
  const DF r = df_add(sm[warp], ex);
  *total = sm[32];
  sync();
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

// Draft logits of columns [v0, v0 + n) (n <= 64) into zs[], using all `nthreads` threads (a
// multiple of 64). bf16 weights: a split-K dot product (nthreads / 64 threads per column,
// 16-byte loads, shuffle reduction); fp32 weights: the canonical fp32 chain, one thread per
// column.
template <int UDT, int WDT, class Sync>
__device__ void segment_logits(const RowJob& j, const RowInfo& ri, int v0, int n, float* zs,
                               int tid, int nthreads, Sync sync) {
  if (WDT == SPEC_BF16 && j.rank > 0 && (j.rank % 8) == 0) {
    const int tpc = nthreads / 64;  // threads per column
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
  sync();
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void l2_prefetch_bytes(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Select of row `row` (row info `ri`) by threads tid = 0 .. nthreads-1 (a multiple of 64, at
// most 1024, starting at a warp boundary), which synchronise with `sync`:
//   kind 0 (MODE_STATS partials): greedy argmax, or inverse-CDF draw from the softmax;
//   kind 1 (MODE_RESID partials): inverse-CDF draw from the residual / bonus distribution.
// Only the crossing segment is recomputed element by element; everything else uses the
// partials. Markov segments (<= 64 columns) are rebuilt once into shared memory.
template <int UDT, int WDT, bool COHERENT, class Sync>
__device__ void select_row(const RowJob& j, const RowInfo& ri, int row, int seg, int nseg,
                           const float* pm, const float* ps, const int* pi, const SelectOut& o,
                           int tid, int nthreads, Sync sync, SelectShared& S) {
  const bool resid = o.kind == 1;
  const float u_row = (o.greedy && !resid) ? 0.0f : o.uni[(size_t)row * o.uni_stride + o.uni_offset];
  const bool markov = resid ? (ri.resid && j.rank > 0) : j.rank > 0;
  const bool need_z = j.rank > 0 && (!resid || ri.resid);

  // 1. normaliser from the partials. Warp w owns the contiguous segment range [s0, s1) of the
  // row's (row-major) partials and lane l a contiguous run [c0, c1) of it; a run of up to kPer
  // segments stays in registers through the crossing search below.
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
  const int s0 = (int)((long long)nseg * warp / nwarps);
  const int s1 = (int)((long long)nseg * (warp + 1) / nwarps);
  const int per = (s1 - s0 + 31) / 32;
  const int c0 = min(s1, s0 + lane * per), c1 = min(s1, c0 + per);
  const float* rpm = pm + (size_t)row * nseg;
  const float* rps = ps + (size_t)row * nseg;
  constexpr int kPer = 16;
  const bool in_regs = per <= kPer;  // the same for every thread of the select
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
          lm[k] = ld_part<COHERENT>(rpm + c);
          ls[k] = ld_part<COHERENT>(rps + c);
          if (rpi) li[k] = ld_part<COHERENT>(rpi + c);
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
        const float v = ld_part<COHERENT>(rpm + c);
        const int ix = rpi ? ld_part<COHERENT>(rpi + c) : 0x7fffffff;
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
    if (lane == 0) {
      S.wm[warp] = lmax;
      S.wi[warp] = lidx;
    }
    sync();
    for (int w = 0; w < nwarps; ++w) {
      const float om = S.wm[w];
      const int oi = S.wi[w];
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
        ls[k] = c0 + k < c1 ? ld_part<COHERENT>(rps + c0 + k) : 0.0f;
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      ls[k] = c0 + k < c1 ? weight(lm[k], ls[k]) : 0.0f;  // ls now holds the weights
      lsum = df_add(lsum, ls[k]);
    }
  } else {
    for (int c = c0; c < c1; ++c)
      lsum = df_add(lsum, weight(resid ? 0.0f : ld_part<COHERENT>(rpm + c),
                                 ld_part<COHERENT>(rps + c)));
  }
  const DF incl = warp_scan_df(lsum);
  DF run_before = df_shfl_up(incl, 1);  // the warp's mass before this run
  if (lane == 0) run_before = df_zero();
  if (lane == 31) S.wt[warp] = incl;
  sync();
  DF Z = df_zero();
  for (int w = 0; w < nwarps; ++w) Z = df_add(Z, S.wt[w]);
  if (tid == 0) {
    S.M = M;
    const bool zok = Z.hi > 0.0f && isfinite(Z.hi);
    S.lz = resid ? 0.0f : (zok ? df_log(Z) : logf(Z.hi));
    S.c = -1;
    S.rem = 0.0f;
    S.x = -1;
    S.last = -1;
    S.zv0 = -1;
    if (!resid && (!zok || !(M > -INFINITY))) atomicOr(j.status, SPEC_DEV_NONFINITE);
  }
  sync();

  int x = -1;
  if (!resid && o.greedy) {
    x = gidx;
    if (x < 0 || x >= j.V) {
      if (tid == 0) atomicOr(j.status, SPEC_DEV_NONFINITE);
      x = 0;
    }
    if (markov && o.logp) {  // rebuild the segment holding x for its log-probability
      const int v0 = (x / 64) * 64;
      segment_logits<UDT, WDT>(j, ri, v0, min(64, j.V - v0), S.zs, tid, nthreads, sync);
      if (tid == 0) S.zv0 = v0;
      sync();
    }
  } else {
    // 3. crossing segment for t = u * Z: the warp whose mass holds t, the first lane of it
    // whose cumulative mass exceeds t, then that lane's run in order
    const DF t = df_mul(Z, u_row);
    DF before = df_zero();
    int wstar = -1;
    for (int w = 0; w < nwarps; ++w) {
      const DF next = df_add(before, S.wt[w]);
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
            const float wv = weight(resid ? 0.0f : ld_part<COHERENT>(rpm + c),
                                    ld_part<COHERENT>(rps + c));
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
        S.c = found >= 0 ? found : lastpos;
        S.rem = found >= 0 ? remv : 1e30f;
      }
    }
    sync();
    if (S.c < 0 && tid == 0) {
      // rounding left no crossing: the end of the last segment with positive mass
      int last = -1;
      for (int c = nseg - 1; c >= 0 && last < 0; --c)
        if (ld_part<COHERENT>(rps + c) > 0.0f) last = c;
      if (last < 0) atomicOr(j.status, resid ? SPEC_DEV_EMPTY_RESIDUAL : SPEC_DEV_NONFINITE);
      S.c = last;
      S.rem = 1e30f;
    }
    sync();
    const int cstar = S.c;
    const float rem = S.rem;
    Norm dn = {0.0f, 0.0f}, tn = {0.0f, 0.0f};
    if (resid) {
      if (ri.trow >= 0 && j.tstats) tn = load_norm(j.tstats, ri.trow);
      if (ri.urow >= 0 && j.dstats) dn = load_norm(j.dstats, ri.urow);
    }
    const int v0 = max(cstar, 0) * seg, v1 = min(j.V, v0 + seg);
    if (seg <= 64) {
      // 3a. small segment: values into shared memory, warp 0 scans in token order
      if (need_z) {
        segment_logits<UDT, WDT>(j, ri, v0, v1 - v0, S.zs, tid, nthreads, sync);
        if (tid == 0) S.zv0 = v0;
      }
      for (int e = tid; e < v1 - v0; e += nthreads) {
        const float zd = need_z ? S.zs[e] : (ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v0 + e) : 0.0f);
        S.es[e] = seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v0 + e, zd);
      }
      sync();
      if (tid < 32 && cstar >= 0) {
        const int n = v1 - v0;
        float a0 = tid < n ? S.es[tid] : 0.0f, a1 = tid + 32 < n ? S.es[tid + 32] : 0.0f;
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
          if (m0) S.x = v0 + __ffs(m0) - 1;
          else if (m1) S.x = v0 + 32 + __ffs(m1) - 1;
          S.last = p1 ? v0 + 32 + 31 - __clz(p1) : (p0 ? v0 + 31 - __clz(p0) : -1);
        }
      }
    } else {
      // 3b. long segment (no Markov bias): per-thread runs, block scan, rescan one run
      const int per = (seg + nthreads - 1) / nthreads;
      const int e0 = min(v1, v0 + tid * per), e1 = min(v1, e0 + per);
      DF mine = df_zero();
      for (int v = e0; v < e1; ++v)
        mine = df_add(mine, seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                                ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f));
      DF segtot;
      const DF sbefore = block_exscan_df(mine, &segtot, tid, nthreads, sync, S.scan);
      const DF r = {rem, 0.0f};
      if (cstar >= 0) {
        if (!df_gt(sbefore, r) && df_gt(df_add(sbefore, mine), r)) {
          DF cum = sbefore;
          for (int v = e0; v < e1; ++v) {
            const float w = seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                                ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f);
            cum = df_add(cum, w);
            if (df_gt(cum, r)) {
              S.x = v;
              break;
            }
          }
        }
        int lastp = -1;
        for (int v = e1 - 1; v >= e0 && lastp < 0; --v)
          if (seg_value<UDT, WDT>(j, ri, resid, M, dn, tn, v,
                                  ri.urow >= 0 ? draft_logit<UDT, WDT>(j, ri, v) : 0.0f) > 0.0f)
            lastp = v;
        if (lastp >= 0) atomicMax(&S.last, lastp);
      }
    }
    sync();
    x = S.x >= 0 ? S.x : S.last;
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
      // the row's (request, position): its draft base-logit row
      const size_t q = (size_t)ri.urow;
      o.tokens[q] = x;
      if (o.w1) l2_prefetch_bytes(static_cast<const char*>(o.w1) + (size_t)x * o.w1_row_bytes,
                                  o.w1_row_bytes);
      if (o.logp) {
        const int zv0 = S.zv0;
        const float zx = (zv0 >= 0 && x >= zv0 && x < zv0 + 64) ? S.zs[x - zv0]
                                                                : draft_logit<UDT, WDT>(j, ri, x);
        o.logp[q] = zx - S.M - S.lz;
      }
      if (o.stats) {
        o.stats[2 * q] = S.M;
        o.stats[2 * q + 1] = S.lz;
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

}  // namespace spec
