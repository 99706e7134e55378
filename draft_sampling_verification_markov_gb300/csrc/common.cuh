// common.cuh -- device helpers shared by the kernels of libspecmarkov.
//
// Row jobs. Every pass of the hot path walks a set of logit rows and, per row, a segment of the
// vocabulary at a time. A row job says, for row m of the pass, which draft base-logit row,
// which target row and which previous token (for the Markov bias) it reads, and with which
// normalisers. Producers (the streaming kernels, the generic FFMA kernel and the tcgen05
// kernel) reduce each (row, segment) to a partial; consumers (select / finalize kernels)
// combine the partials of a row.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_markov.h"

namespace spec {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------------------ launch chaining

// Programmatic dependent launch. A kernel launched with programmatic stream serialisation is
// scheduled as the blocks of the kernel before it on the stream exit, without waiting for that
// kernel's completion and memory flush. grid_dep_wait() returns once that kernel has completed
// and its writes are visible; a thread must pass it before it reads anything the earlier kernels
// of the call write, or writes anything they read. For a kernel launched without the attribute
// it returns at once. No kernel here signals its dependents early
// (griddepcontrol.launch_dependents): a Markov pass scheduled while the select kernel still ran
// made every such pair about 6 us slower, even with nothing done before its wait.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------------------ element loads

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Element i of an f32 (DT == SPEC_F32) or bf16 (DT == SPEC_BF16) array, as fp32.
template <int DT>
__device__ __forceinline__ float ld_elem(const void* p, size_t i) {
  if constexpr (DT == SPEC_BF16) {
    return bf16_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
  } else {
    return __ldg(reinterpret_cast<const float*>(p) + i);
  }
}

// Streaming (read-once) 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// exp2 on the MUFU pipe (ex2.approx, flush-to-zero): max relative error ~2^-22.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(z - m) as 2^((z - m) * log2 e). The subtraction comes first so that the row maximum maps
// to exactly 1 (folding m into an FMA would scale every term by the rounding error of
// m * log2 e, which compounds when partials are merged).
__device__ __forceinline__ float exp_shift(float z, float m) {
  return fast_exp2((z - m) * kLog2e);
}

// ------------------------------------------------------------------------------ softmax partials

// (max, sum of exp(z - max), index of the first maximum) over a set of values.
struct StatsAcc {
  float m;
  float s;
  int idx;
};

__device__ __forceinline__ StatsAcc stats_empty() { return {-INFINITY, 0.0f, 0x7fffffff}; }

// Merge two partials; ties of the maximum keep the lower index.
__device__ __forceinline__ StatsAcc stats_merge(StatsAcc a, StatsAcc b) {
  StatsAcc o;
  o.m = fmaxf(a.m, b.m);
  if (o.m == -INFINITY) {
    o.s = 0.0f;
  } else {
    o.s = (a.s == 0.0f ? 0.0f : a.s * exp_shift(a.m, o.m)) +
          (b.s == 0.0f ? 0.0f : b.s * exp_shift(b.m, o.m));
  }
  if (a.m > b.m || (a.m == b.m && a.idx < b.idx))
    o.idx = a.idx;
  else
    o.idx = b.idx;
  return o;
}

__device__ __forceinline__ StatsAcc warp_merge(StatsAcc a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    StatsAcc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, off);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
    b.idx = __shfl_xor_sync(0xffffffffu, a.idx, off);
    a = stats_merge(a, b);
  }
  return a;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// ------------------------------------------------------------------------------ double-float sums
// Long sums and prefix sums are carried as an unevaluated pair hi + lo of fp32 numbers: Knuth's
// TwoSum yields the exact rounding error of an fp32 addition, so a pair keeps about 48 bits
// while using only fp32 arithmetic (fp64 runs at a small fraction of the fp32 rate here).
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_zero() { return {0.0f, 0.0f}; }

// s + e == a + b exactly, s = fl(a + b) (Knuth, TAOCP vol. 2, 4.2.2).
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// The same when |a| >= |b| (Dekker).
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DF df_add(DF a, float b) {
  const DF s = two_sum(a.hi, b);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  const DF t = two_sum(a.lo, b.lo);
  const DF u = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return fast_two_sum(u.hi, __fadd_rn(u.lo, t.lo));
}

__device__ __forceinline__ DF df_neg(DF a) { return {-a.hi, -a.lo}; }

// a * b for an fp32 b (the product's rounding error from an fma).
__device__ __forceinline__ DF df_mul(DF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  const float e = fmaf(a.hi, b, -p);
  return fast_two_sum(p, fmaf(a.lo, b, e));
}

// a > b for normalised pairs (|lo| at most half an ulp of hi).
__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ float df_float(DF a) { return __fadd_rn(a.hi, a.lo); }

__device__ __forceinline__ DF df_shfl_xor(DF a, int off) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
}

__device__ __forceinline__ DF df_shfl_up(DF a, int off) {
  return {__shfl_up_sync(0xffffffffu, a.hi, off), __shfl_up_sync(0xffffffffu, a.lo, off)};
}

__device__ __forceinline__ DF df_shfl(DF a, int lane) {
  return {__shfl_sync(0xffffffffu, a.hi, lane), __shfl_sync(0xffffffffu, a.lo, lane)};
}

// Warp sum; df_add is commutative, so every lane receives the same pair.
__device__ __forceinline__ DF warp_sum_df(DF x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = df_add(x, df_shfl_xor(x, off));
  return x;
}

// Inclusive warp prefix sum in lane order.
__device__ __forceinline__ DF warp_scan_df(DF x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const DF y = df_shfl_up(x, off);
    if (lane >= off) x = df_add(y, x);
  }
  return x;
}

// log(hi + lo) for a positive normalised pair.
__device__ __forceinline__ float df_log(DF a) { return logf(a.hi) + a.lo / a.hi; }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

// Block-wide merge through shared memory (blockDim.x a multiple of 32, <= 1024). All threads
// receive the result.
__device__ __forceinline__ StatsAcc block_merge(StatsAcc a) {
  __shared__ float sm_m[32];
  __shared__ float sm_s[32];
  __shared__ int sm_i[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  a = warp_merge(a);
  __syncthreads();
  if (lane == 0) {
    sm_m[warp] = a.m;
    sm_s[warp] = a.s;
    sm_i[warp] = a.idx;
  }
  __syncthreads();
  StatsAcc b = stats_empty();
  if (lane < nw) b = {sm_m[lane], sm_s[lane], sm_i[lane]};
  b = warp_merge(b);
  return b;
}

__device__ __forceinline__ float block_sum(float x) {
  __shared__ float sm[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  x = warp_sum(x);
  __syncthreads();
  if (lane == 0) sm[warp] = x;
  __syncthreads();
  float y = lane < nw ? sm[lane] : 0.0f;
  return warp_sum(y);
}

// ------------------------------------------------------------------------------ row jobs

// How row m of a pass maps onto the problem.
enum RowMap : int {
  MAP_POSITION = 0,  // m = r, draft position k fixed (propose step k)
  MAP_ALL_POS = 1,   // m = r*gamma + (k-1), every draft position (TV, draft stats)
  MAP_FINAL = 2,     // m = r, the final row n_r of rejection verification
  MAP_TARGET = 3,    // m = r*(gamma+1) + i, target rows only
};

// What a pass reduces per (row, segment).
enum PassMode : int {
  MODE_STATS = 0,  // softmax partials (max, sum exp, argmax) of the draft or target logits
  MODE_RESID = 1,  // sum of max(0, p_t - p_d) (p_d == 0 for the bonus row)
  MODE_TV = 2,     // sum of min(p_d, p_t)
};

struct RowJob {
  int rows;          // rows in the pass
  int map;           // RowMap
  int mode;          // PassMode
  int R, gamma, V;
  int k;             // draft position (MAP_POSITION)
  float scale;       // multiplier applied to the logits (1/T, or 1 for greedy)
  // draft side
  const void* U;     // [R, gamma, V]
  const void* W1;    // [V, rank]
  const void* W2;    // [V, rank]
  int rank;
  const int32_t* anchors;  // [R]
  const int32_t* tokens;   // [R, gamma] proposed tokens
  const float* dstats;     // [R, gamma, 2] draft (m, log Z)
  // target side
  const void* T;           // [R, gamma+1, V]
  const float* tstats;     // [R*(gamma+1), 2] target (m, log Z)
  const int32_t* lengths;  // [R] or null
  const int32_t* final_n;  // [R] n_r (MAP_FINAL)
  const int32_t* final_kind;  // [R] 1 = residual, 0 = bonus (MAP_FINAL)
  uint32_t* status;
  // grammar-masked drafting: allowed draft tokens [R, mask_words] (bit v%32 of word v/32), or
  // null for no mask; a disallowed token has draft logit -inf
  const uint32_t* mask;
  int mask_words;
  // flattened verify batch: target rows of request r are toff[r] .. toff[r+1]-1 of a packed
  // [*, V] array (toff[R] rows in all), or null for the padded [R, gamma+1, V] layout
  const int32_t* toff;
  // nonzero: the pass may be launched while the previous kernel of the same call still runs
  // (its kernels then wait with grid_dep_wait before touching that kernel's data)
  int pdl;
};

// Row of target position i (0..gamma) of request r in a target array of R*(gamma+1) rows,
// padded (toff null) or flattened. A flattened row outside the array (offsets that do not
// match the lengths) is flagged and read as row 0, so no access leaves the array.
__device__ __forceinline__ long long target_row(const int32_t* toff, int R, int gamma, int r,
                                                int i, uint32_t* status) {
  const long long g1 = (long long)gamma + 1;
  if (!toff) return (long long)r * g1 + i;
  const long long t = (long long)toff[r] + i;
  if (t < 0 || t >= (long long)R * g1) {
    atomicOr(status, SPEC_DEV_BAD_LENGTH);
    return 0;
  }
  return t;
}
__device__ __forceinline__ long long target_row(const RowJob& j, int r, int i) {
  return target_row(j.toff, j.R, j.gamma, r, i, j.status);
}

// Whether request r may propose token v.
__device__ __forceinline__ bool draft_allowed(const RowJob& j, int r, int v) {
  return !j.mask || ((j.mask[(size_t)r * j.mask_words + (v >> 5)] >> (v & 31)) & 1u);
}

struct RowInfo {
  int active;   // 0: the row is not needed (beyond the verified length)
  int r;
  long long urow;  // draft base-logit row index into [R*gamma, V] (-1: none)
  long long trow;  // target row index into [R*(gamma+1), V] (-1: none)
  int prev;        // previous token for the Markov bias (-1: none)
  int resid;       // MODE_RESID: 1 residual, 0 bonus
};

__device__ __forceinline__ int checked_token(const RowJob& j, int t) {
  if (t < 0 || t >= j.V) {
    atomicOr(j.status, SPEC_DEV_BAD_TOKEN);
    return 0;
  }
  return t;
}

__device__ __forceinline__ int checked_length(const RowJob& j, int r) {
  if (!j.lengths) return j.gamma;
  int l = j.lengths[r];
  if (l < 0 || l > j.gamma) {
    atomicOr(j.status, SPEC_DEV_BAD_LENGTH);
    l = l < 0 ? 0 : j.gamma;
  }
  return l;
}

__device__ __forceinline__ RowInfo row_info(const RowJob& j, int m) {
  RowInfo o;
  o.active = 1;
  o.urow = -1;
  o.trow = -1;
  o.prev = -1;
  o.resid = 0;
  const int g = j.gamma;
  switch (j.map) {
    case MAP_POSITION: {
      o.r = m;
      o.urow = (long long)m * g + (j.k - 1);
      if (j.rank > 0)
        o.prev = checked_token(j, j.k == 1 ? j.anchors[m] : j.tokens[(size_t)m * g + j.k - 2]);
      break;
    }
    case MAP_ALL_POS: {
      const int r = m / g, k = m % g + 1;
      o.r = r;
      o.urow = m;
      o.trow = target_row(j, r, k - 1);
      if (j.rank > 0) o.prev = checked_token(j, k == 1 ? j.anchors[r] : j.tokens[(size_t)m - 1]);
      break;
    }
    case MAP_FINAL: {
      const int r = m, n = j.final_n[r];
      o.r = r;
      o.trow = target_row(j, r, n);
      o.resid = j.final_kind[r];
      if (o.resid) {
        o.urow = (long long)r * g + n;
        if (j.rank > 0)
          o.prev = checked_token(j, n == 0 ? j.anchors[r] : j.tokens[(size_t)r * g + n - 1]);
      }
      break;
    }
    default: {  // MAP_TARGET
      o.trow = m;
      if (j.toff) {  // flattened: the first toff[R] rows are the batch
        o.r = 0;      // target rows have no draft side
        o.active = m < j.toff[j.R];
        break;
      }
      const int r = m / (g + 1), i = m % (g + 1);
      o.r = r;
      if (j.lengths) o.active = i <= checked_length(j, r);
      break;
    }
  }
  return o;
}

// Row normaliser: p(v) = exp(z(v) - m - log Z).
struct Norm {
  float m;
  float lz;
};

__device__ __forceinline__ Norm load_norm(const float* stats, long long row) {
  return {stats[2 * row], stats[2 * row + 1]};
}

// Probability from a (scaled) logit and its row normaliser; z - m first (exact near the mode).
__device__ __forceinline__ float prob_of(float z, Norm n) {
  return fast_exp2(((z - n.m) - n.lz) * kLog2e);
}

// ------------------------------------------------------------------------------ workspace

// Byte layout of a caller workspace, identical for spec_workspace_bytes and every op.
struct WsLayout {
  size_t header;       // 256 bytes: status word + spare
  size_t off_pm, off_ps, off_pi;  // partials (max / sum / argmax)  [nseg][rows]
  size_t off_tstats;   // [R*(gamma+1), 2]
  size_t off_dstats;   // [R*gamma, 2]
  size_t off_final;    // [R] n, [R] kind
  size_t total;
};

}  // namespace spec
