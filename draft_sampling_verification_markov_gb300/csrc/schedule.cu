// schedule.cu -- hardware-aware prefix scheduler ("[DeepSeek-6] DSpark", section 6).
//
// Maximise Theta = tau * SPS(B) over the verify lengths l_r, with B = sum(1 + l_r) and
// tau = sum(1 + sum_{j<=l_r} a_{r,j}). Every candidate (r, j) is queued by a_{r,j} in decreasing
// order (ties: r ascending, then j ascending); because a is non-increasing in j, every queue
// prefix is prefix-closed per request, and for a fixed B = R + K the first K candidates give the
// largest tau. Scanning K therefore finds the optimum.
//
// One CTA does everything in shared memory (R * gamma <= 16384 candidates):
//   1. keys = (~bits(a) << 32) | (r * gamma + j - 1), sorted ascending by a bitonic network;
//   2. q = round-half-even(a * 2^32) per sorted candidate, an exact uint64 inclusive scan S_K;
//   3. Theta(K) = double(R * 2^32 + S_K) * sps[R + K], arg-max with the smallest K on ties;
//   4. l_r = number of selected candidates of request r.
// The integer prefix sums and the single IEEE multiply make the result independent of the
// summation order, so it is bit-identical to any implementation of the same definition.
//
// Dynamic top-K (section 7): with a device-resident capacity B_cap (a batch size decided from an
// earlier step's confidences) the selection is K = clamp(B_cap - R, 0, Kmax), the first K
// candidates of the current queue, and Theta(K) is reported for that K. The search of step 3 still
// runs on the same sorted queue, and its optimum R + K* can be written out as the capacity of a
// later step, so one sort serves both.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {

constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* survival,
                                                                 const double* sps, int Bmax,
                                                                 int R, int gamma, int npow2,
                                                                 const int32_t* b_cap,
                                                                 int32_t* lengths, int32_t* B_out,
                                                                 double* theta_out,
                                                                 int32_t* B_opt_out,
                                                                 uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);  // [npow2]
  int* len = reinterpret_cast<int*>(key + npow2);                       // [R]
  __shared__ unsigned long long warp_tot[32];
  __shared__ double best_theta[32];
  __shared__ int best_k[32];
  __shared__ double fixed_theta;

  const int n = R * gamma;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // 1. keys
  for (int i = tid; i < npow2; i += blockDim.x) {
    unsigned long long k = ~0ull;
    if (i < n) {
      float a = survival[i];
      if (!(a >= 0.0f && a <= 1.0f)) {  // NaN or out of range: flag and clamp
        atomicOr(status, SPEC_DEV_NONFINITE);
        a = a > 1.0f ? 1.0f : 0.0f;
      }
      uint32_t bits = __float_as_uint(a) & 0x7fffffffu;  // +0 and -0 alike
      k = ((unsigned long long)(~bits) << 32) | (unsigned long long)i;
    }
    key[i] = k;
  }
  for (int r = tid; r < R; r += blockDim.x) len[r] = 0;
  __syncthreads();

  // bitonic sort, ascending
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < (npow2 >> 1); t += blockDim.x) {
        const int lo = (t / stride) * stride * 2 + (t % stride);
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = key[lo], y = key[hi];
        if ((x > y) == up) {
          key[lo] = y;
          key[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  // 2. fixed-point prefix sums over the sorted queue; thread t owns sorted slots
  //    [t*per, (t+1)*per)
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int s0 = min(n, tid * per), s1 = min(n, s0 + per);
  auto q_of = [&](int slot) -> unsigned long long {
    const uint32_t bits = ~(uint32_t)(key[slot] >> 32);
    const float a = __uint_as_float(bits);
    return (unsigned long long)__double2ull_rn((double)a * 4294967296.0);
  };
  unsigned long long local = 0;
  for (int s = s0; s < s1; ++s) local += q_of(s);
  unsigned long long inc = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    unsigned long long w = lane < nw ? warp_tot[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
  }
  __syncthreads();
  unsigned long long S = warp_tot[warp] + inc - local;  // exclusive prefix of this thread

  // 3. Theta(K) for K in [0, Kmax]; thread t evaluates K = slot + 1 for its slots (and K = 0)
  const int Kmax = min(n, Bmax - R);
  const unsigned long long base = (unsigned long long)R << 32;
  int Kcap = -1;  // fixed K of the dynamic top-K, -1 for the Theta search
  if (b_cap) {
    const int cap = *b_cap;
    if (cap < 0 && tid == 0) atomicOr(status, SPEC_DEV_BAD_LENGTH);
    const long long want = (long long)cap - R;
    Kcap = want <= 0 ? 0 : (want < Kmax ? (int)want : Kmax);
  }
  double bt = -1.0;
  int bk = 0x7fffffff;
  if (tid == 0) {
    bt = (double)base * sps[R];
    bk = 0;
    if (Kcap == 0) fixed_theta = bt;
  }
  for (int s = s0; s < s1; ++s) {
    S += q_of(s);
    const int K = s + 1;
    if (K > Kmax) break;
    const double th = (double)(base + S) * sps[R + K];
    if (K == Kcap) fixed_theta = th;  // exactly one thread holds slot Kcap - 1
    if (th > bt) {  // slots ascend, so the first maximum in this run has the smallest K
      bt = th;
      bk = K;
    }
  }
  // block arg-max: larger Theta wins, ties go to the smaller K
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double ot = __shfl_xor_sync(0xffffffffu, bt, off);
    const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
    if (ot > bt || (ot == bt && ok < bk)) {
      bt = ot;
      bk = ok;
    }
  }
  if (lane == 0) {
    best_theta[warp] = bt;
    best_k[warp] = bk;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    bt = lane < nw ? best_theta[lane] : -1.0;
    bk = lane < nw ? best_k[lane] : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const double ot = __shfl_xor_sync(0xffffffffu, bt, off);
      const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
      if (ot > bt || (ot == bt && ok < bk)) {
        bt = ot;
        bk = ok;
      }
    }
    if (lane == 0) {
      best_theta[0] = bt;
      best_k[0] = bk;
    }
  }
  __syncthreads();
  const int Kstar = best_k[0];
  const int Ksel = Kcap >= 0 ? Kcap : Kstar;

  // 4. lengths
  for (int s = tid; s < Ksel; s += blockDim.x) {
    const int idx = (int)(key[s] & 0xffffffffull);
    atomicAdd(&len[idx / gamma], 1);
  }
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) lengths[r] = len[r];
  if (tid == 0) {
    *B_out = R + Ksel;
    *theta_out = (Kcap >= 0 ? fixed_theta : best_theta[0]) / 4294967296.0;
    if (B_opt_out) *B_opt_out = R + Kstar;
  }
}

size_t schedule_smem_bytes(int R, int gamma) {
  int n = R * gamma, p = 1;
  while (p < n) p <<= 1;
  return (size_t)p * 8 + (size_t)R * 4;
}

cudaError_t launch_schedule(const float* survival, const double* sps, int Bmax, int R, int gamma,
                            const int32_t* b_cap, int32_t* lengths, int32_t* B_out,
                            double* theta_out, int32_t* B_opt_out, uint32_t* status,
                            cudaStream_t s) {
  int n = R * gamma, p = 1;
  while (p < n) p <<= 1;
  if (p < 2) p = 2;
  const size_t smem = (size_t)p * 8 + (size_t)R * 4;
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, s>>>(survival, sps, Bmax, R, gamma, p, b_cap, lengths,
                                                 B_out, theta_out, B_opt_out, status);
  return cudaGetLastError();
}

// Flattened verify batch ("[DeepSeek-6] DSpark", section 7: physical execution decoupled from
// the logical sequences, with a marker tensor carrying the per-sequence structure): request r
// owns the 1 + l_r packed target rows offsets[r] .. offsets[r+1]-1 (positions 0..l_r), and the
// markers give each packed row its request and position (-1 past the batch). One CTA: every
// thread sums a contiguous run of requests, a block scan gives each run its first row.
__global__ void __launch_bounds__(kSchedThreads) flat_layout_kernel(const int32_t* lengths, int R,
                                                                    int gamma, int32_t* offsets,
                                                                    int32_t* row_req,
                                                                    int32_t* row_pos,
                                                                    uint32_t* status) {
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto len = [&](int r) {
    int l = lengths[r];
    if (l < 0 || l > gamma) {
      atomicOr(status, SPEC_DEV_BAD_LENGTH);
      l = l < 0 ? 0 : gamma;
    }
    return l;
  };
  const int per = (R + blockDim.x - 1) / blockDim.x;
  const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += 1 + len(r);
  int inc = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
    if (lane == 31) total = wi;
  }
  __syncthreads();
  int S = warp_tot[warp] + inc - local;  // first packed row of this thread's requests
  for (int r = r0; r < r1; ++r) {
    const int l = len(r);
    offsets[r] = S;
    if (row_req)
      for (int i = 0; i <= l; ++i) row_req[S + i] = r;
    if (row_pos)
      for (int i = 0; i <= l; ++i) row_pos[S + i] = i;
    S += 1 + l;
  }
  const int B = total;
  if (tid == 0) offsets[R] = B;
  const int cap = R * (gamma + 1);
  for (int b = B + tid; b < cap; b += blockDim.x) {
    if (row_req) row_req[b] = -1;
    if (row_pos) row_pos[b] = -1;
  }
}

// Copy of the verified rows of a padded [R, gamma+1, row] array into the flattened layout:
// padded row (r, i), i <= l_r, to packed row offsets[r] + i. One block per padded row; rows past
// a request's length are neither read nor written, so the bytes moved are those of the B rows.
__global__ void __launch_bounds__(256) flat_pack_kernel(const char* src, int row_bytes,
                                                        const int32_t* lengths,
                                                        const int32_t* offsets, int R, int gamma,
                                                        char* dst, uint32_t* status) {
  const long long row = blockIdx.x;
  const int r = (int)(row / (gamma + 1)), i = (int)(row % (gamma + 1));
  int l = lengths[r];
  if (l < 0 || l > gamma) {
    if (threadIdx.x == 0) atomicOr(status, SPEC_DEV_BAD_LENGTH);
    l = l < 0 ? 0 : gamma;
  }
  if (i > l) return;
  const long long b = (long long)offsets[r] + i;
  if (b < 0 || b >= (long long)R * (gamma + 1)) {
    if (threadIdx.x == 0) atomicOr(status, SPEC_DEV_BAD_LENGTH);
    return;
  }
  const char* from = src + row * row_bytes;
  char* to = dst + b * row_bytes;
  if (row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
    const uint4* f = reinterpret_cast<const uint4*>(from);
    uint4* t = reinterpret_cast<uint4*>(to);
    const int n = row_bytes / 16;
    for (int w = threadIdx.x; w < n; w += 4 * blockDim.x) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int x = w + k * blockDim.x;
        if (x < n) v[k] = ld_stream16(f + x);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int x = w + k * blockDim.x;
        if (x < n) t[x] = v[k];
      }
    }
  } else {  // row_bytes % 4 == 0
    const uint32_t* f = reinterpret_cast<const uint32_t*>(from);
    uint32_t* t = reinterpret_cast<uint32_t*>(to);
    for (int w = threadIdx.x; w < row_bytes / 4; w += blockDim.x) t[w] = f[w];
  }
}

void launch_flat_pack(const void* src, int row_bytes, const int32_t* lengths,
                      const int32_t* offsets, int R, int gamma, void* dst, uint32_t* status,
                      cudaStream_t s) {
  const long long rows = (long long)R * (gamma + 1);
  flat_pack_kernel<<<(unsigned)rows, 256, 0, s>>>(static_cast<const char*>(src), row_bytes,
                                                  lengths, offsets, R, gamma,
                                                  static_cast<char*>(dst), status);
}

void launch_flat_layout(const int32_t* lengths, int R, int gamma, int32_t* offsets,
                        int32_t* row_req, int32_t* row_pos, uint32_t* status, cudaStream_t s) {
  flat_layout_kernel<<<1, kSchedThreads, 0, s>>>(lengths, R, gamma, offsets, row_req, row_pos,
                                                 status);
}

}  // namespace spec
