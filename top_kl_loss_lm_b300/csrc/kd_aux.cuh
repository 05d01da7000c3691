// kd_aux.cuh — the small kernels around the GEMMs:
//   prep     per row: sort the teacher's cached (id, logit) pairs by id, teacher
//            softmax at T, entropy sum_j P_j log P_j of the teacher grid, id check
//   combine  per row: merge the (max, sum) partials into lse, loss = entropy -
//            <P, Z>/T + lse
//   dh sum   per element: sum the k-split partials of dH in fixed order -> bf16
//   wait probe  one bounded wait that nothing satisfies (error-path test)
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_bf16.h>

#include "kd_ptx.cuh"
#include "kd_sched.h"

namespace kd {

constexpr int kPrepWarps = 8;
constexpr int kMaxTopK = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row. Output pairs[row][r] = (id, bits of p) in ascending id order
// (ties keep cache order); masked rows get (INT_MAX, 0) and entropy 0 and their
// inputs are not read. An id outside [0, V) at a counted row records
// KD_ERR_INDEX and is replaced by INT_MAX so no tile ever matches it.
__global__ void __launch_bounds__(kPrepWarps * 32)
    kd_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ t,
                   const uint8_t* __restrict__ mask, int64_t N, int K, int V, float inv_T,
                   int2* __restrict__ pairs, float* __restrict__ ent,
                   unsigned long long* n_valid, int* status) {
  __shared__ int s_key[kPrepWarps][kMaxTopK];
  __shared__ int s_skey[kPrepWarps][kMaxTopK];
  __shared__ float s_sp[kPrepWarps][kMaxTopK];
  __shared__ float s_slogp[kPrepWarps][kMaxTopK];
  __shared__ unsigned int s_count;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_count = 0;
  __syncthreads();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kPrepWarps + warp;
  if (row < N) {
    const bool counted = (mask == nullptr) || (mask[row] != 0);
    int2* out = pairs + row * K;
    if (!counted) {
      for (int k = lane; k < K; k += 32) out[k] = make_int2(INT_MAX, 0);
      if (lane == 0) ent[row] = 0.0f;
    } else {
      if (lane == 0) atomicAdd(&s_count, 1u);
      constexpr int kPer = kMaxTopK / 32;
      int key[kPer];
      float b[kPer];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = lane + 32 * i;
        key[i] = INT_MAX;
        b[i] = -INFINITY;
        if (k < K) {
          int id = idx[row * K + k];
          if (id < 0 || id >= V) {
            atomicCAS(status, 0, 5 /* KD_ERR_INDEX */);
            id = INT_MAX;
          }
          key[i] = id;
          b[i] = t[row * K + k] * inv_T;
          mx = fmaxf(mx, b[i]);
          s_key[warp][k] = id;
        }
      }
      mx = warp_max(mx);
      float se = 0.0f;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i < K) se += expf(b[i] - mx);
      se = warp_sum(se);
      const float lse_b = mx + logf(se);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = lane + 32 * i;
        if (k < K) {
          int rank = 0;
          for (int j = 0; j < K; ++j) {
            const int kj = s_key[warp][j];
            rank += (kj < key[i]) || (kj == key[i] && j < k);
          }
          const float logp = b[i] - lse_b;
          const float p = expf(logp);
          s_skey[warp][rank] = key[i];
          s_sp[warp][rank] = p;
          s_slogp[warp][rank] = logp;
          out[rank] = make_int2(key[i], __float_as_int(p));
        }
      }
      __syncwarp();
      // entropy of the teacher grid: one term per distinct id (repeats merged)
      float e = 0.0f;
      for (int r = lane; r < K; r += 32) {
        const int id = s_skey[warp][r];
        if (id == INT_MAX) continue;
        if (r > 0 && s_skey[warp][r - 1] == id) continue;
        float P = s_sp[warp][r];
        int n = 1;
        for (int r2 = r + 1; r2 < K && s_skey[warp][r2] == id; ++r2, ++n) P += s_sp[warp][r2];
        if (P > 0.0f) e += (n == 1) ? P * s_slogp[warp][r] : P * logf(P);
      }
      e = warp_sum(e);
      if (lane == 0) ent[row] = e;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_count && n_valid)
    atomicAdd(n_valid, static_cast<unsigned long long>(s_count));
}

// One thread per row. Rows of the forward's last row chunk were split over S_last
// vocabulary ranges, all others over S_full.
__global__ void __launch_bounds__(256)
    kd_combine_kernel(int64_t last_start, int S_full, int S_last, const float2* __restrict__ part,
                      int slots,
                      const int2* __restrict__ pairs, const float* __restrict__ zk,
                      const float* __restrict__ ent, const uint8_t* __restrict__ mask, int64_t N,
                      int K, int V, float inv_T, float* __restrict__ loss,
                      float* __restrict__ lse_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= N) return;
  const int S = row >= last_start ? S_last : S_full;  // vocabulary splits of the row's chunk
  float m = -INFINITY, s = 0.0f;
  for (int sl = 0; sl < S; ++sl) {
    const float2 ps = part[row * slots + sl];
    const float mn = fmaxf(m, ps.x);
    s = s * exp2f(m - mn) + ps.y * exp2f(ps.x - mn);
    m = mn;
  }
  const double lse = (static_cast<double>(m) + static_cast<double>(log2f(s))) * 0.6931471805599453;
  lse_out[row] = static_cast<float>(lse);
  const bool counted = (mask == nullptr) || (mask[row] != 0);
  if (!counted) {
    loss[row] = 0.0f;
    return;
  }
  double cross = 0.0;
  for (int k = 0; k < K; ++k) {
    const int2 pr = pairs[row * K + k];
    if (pr.x < V) cross += static_cast<double>(__int_as_float(pr.y)) * static_cast<double>(zk[row * K + k]);
  }
  loss[row] = static_cast<float>(static_cast<double>(ent[row]) - cross * static_cast<double>(inv_T) + lse);
}

// dH[r][c] = bf16(sum_s part[s][r][c]) for r < rows; 8 columns per thread.
__global__ void __launch_bounds__(256)
    kd_dh_sum_kernel(const float* __restrict__ part, int KS, int64_t part_stride, int64_t rows, int D,
                     uint16_t* __restrict__ dH) {
  const int64_t groups = rows * (D / 8);
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups;
       gi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t off = gi * 8;
    float acc[8];
    {
      const float4 a = *reinterpret_cast<const float4*>(part + off);
      const float4 b = *reinterpret_cast<const float4*>(part + off + 4);
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
      acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
    for (int s = 1; s < KS; ++s) {
      const float4 a = *reinterpret_cast<const float4*>(part + s * part_stride + off);
      const float4 b = *reinterpret_cast<const float4*>(part + s * part_stride + off + 4);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    uint4 w;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(acc[0], acc[1]); w.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[2], acc[3]); w.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[4], acc[5]); w.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(acc[6], acc[7]); w.w = *reinterpret_cast<uint32_t*>(&h);
    *reinterpret_cast<uint4*>(dH + off) = w;
  }
}

// A single bounded wait on a barrier that nothing arrives on.
__global__ void kd_wait_probe_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(&bar, 0, &abort_flag, timeout_ns, status, 6 /* KD_ERR_TIMEOUT */);
}

}  // namespace kd
