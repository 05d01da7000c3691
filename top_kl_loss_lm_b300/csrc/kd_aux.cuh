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

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row. The teacher softmax and the entropy of its grid use all K
// entries; the output list pairs[row] holds the entries whose id falls in this
// call's vocabulary range [v0, v0 + Vs) as (id - v0, bits of p) in ascending id
// order (ties keep cache order), followed by (INT_MAX, 0) for the others. The
// whole vocabulary is v0 = 0, Vs = V. Masked rows get (INT_MAX, 0) throughout
// and entropy 0 and their inputs are not read. An id outside [0, V) at a
// counted row records KD_ERR_INDEX and is replaced by INT_MAX so no tile ever
// matches it.
__global__ void __launch_bounds__(kPrepWarps * 32)
    kd_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ t,
                   const uint8_t* __restrict__ mask, int64_t N, int K, int V, int v0, int Vs,
                   float inv_T, int2* __restrict__ pairs, float* __restrict__ ent,
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
      // entries with an id below the range / below its end: the range's entries are
      // sorted positions [lo, hi) and move to the front of the output list
      int below = 0, inside = 0;
      for (int j = lane; j < K; j += 32) {
        const int kj = s_key[warp][j];
        below += kj < v0;
        inside += kj >= v0 && kj - v0 < Vs;
      }
      const int lo = warp_sum_int(below);
      const int n_in = warp_sum_int(inside);
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
          const bool in = rank >= lo && rank < lo + n_in;
          const int pos = in ? rank - lo : (rank < lo ? n_in + rank : rank);
          out[pos] = in ? make_int2(key[i] - v0, __float_as_int(p)) : make_int2(INT_MAX, 0);
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
// vocabulary ranges, all others over S_full. V is the width of the call's
// vocabulary range (the gathered entries are those with a local id below it).
// With shard_out set (a vocabulary shard), the row's (lse over the shard,
// sum_k P_k z_k over the shard's teacher entries) goes there instead of loss /
// lse, for kd_shard_merge_kernel to combine across shards.
__global__ void __launch_bounds__(256)
    kd_combine_kernel(int64_t last_start, int S_full, int S_last, const float2* __restrict__ part,
                      int slots,
                      const int2* __restrict__ pairs, const float* __restrict__ zk,
                      const float* __restrict__ ent, const uint8_t* __restrict__ mask, int64_t N,
                      int K, int V, float inv_T, float* __restrict__ loss,
                      float* __restrict__ lse_out, float2* __restrict__ shard_out) {
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
  const bool counted = (mask == nullptr) || (mask[row] != 0);
  double cross = 0.0;
  if (counted) {
    for (int k = 0; k < K; ++k) {
      const int2 pr = pairs[row * K + k];
      if (pr.x < V)
        cross += static_cast<double>(__int_as_float(pr.y)) * static_cast<double>(zk[row * K + k]);
    }
  }
  if (shard_out != nullptr) {
    shard_out[row] = make_float2(static_cast<float>(lse), static_cast<float>(cross));
    return;
  }
  lse_out[row] = static_cast<float>(lse);
  loss[row] = counted ? static_cast<float>(static_cast<double>(ent[row]) -
                                           cross * static_cast<double>(inv_T) + lse)
                      : 0.0f;
}

// One thread per row: the loss and lse of the whole vocabulary from R shards'
// (lse_r, x_r) pairs (parts[r * N + row]): lse = log sum_r exp(lse_r) and
// loss = entropy - (sum_r x_r) / T + lse at counted rows, 0 elsewhere. The
// shards are combined in index order, so every rank that merges the same
// gathered parts gets the same bits.
__global__ void __launch_bounds__(256)
    kd_shard_merge_kernel(const float2* __restrict__ parts, int R, const float* __restrict__ ent,
                          const uint8_t* __restrict__ mask, int64_t N, float inv_T,
                          float* __restrict__ loss, float* __restrict__ lse_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= N) return;
  double m = -INFINITY;
  for (int r = 0; r < R; ++r) m = fmax(m, static_cast<double>(parts[r * N + row].x));
  double se = 0.0, x = 0.0;
  for (int r = 0; r < R; ++r) {
    const float2 pr = parts[r * N + row];
    se += exp(static_cast<double>(pr.x) - m);
    x += static_cast<double>(pr.y);
  }
  const double lse = m + log(se);
  lse_out[row] = static_cast<float>(lse);
  const bool counted = (mask == nullptr) || (mask[row] != 0);
  loss[row] = counted ? static_cast<float>(static_cast<double>(ent[row]) -
                                           x * static_cast<double>(inv_T) + lse)
                      : 0.0f;
}

// dH[r][c] = sum_s part[s][r][c] for r < rows, summed in split order; 8 columns
// per thread. Written as bf16 (OUT_F32 false) or fp32, the fp32 form optionally
// added to what dH holds (a vocabulary shard's partial dH).
template <bool OUT_F32>
__global__ void __launch_bounds__(256)
    kd_dh_sum_kernel(const float* __restrict__ part, int KS, int64_t part_stride, int64_t rows, int D,
                     void* __restrict__ out, int accumulate) {
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
    if constexpr (OUT_F32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + off);
      float4 lo = make_float4(acc[0], acc[1], acc[2], acc[3]);
      float4 hi = make_float4(acc[4], acc[5], acc[6], acc[7]);
      if (accumulate) {
        const float4 a = o[0], b = o[1];
        lo = make_float4(a.x + lo.x, a.y + lo.y, a.z + lo.z, a.w + lo.w);
        hi = make_float4(b.x + hi.x, b.y + hi.y, b.z + hi.z, b.w + hi.w);
      }
      o[0] = lo;
      o[1] = hi;
    } else {
      uint4 w;
      __nv_bfloat162 h;
      h = __floats2bfloat162_rn(acc[0], acc[1]); w.x = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[2], acc[3]); w.y = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[4], acc[5]); w.z = *reinterpret_cast<uint32_t*>(&h);
      h = __floats2bfloat162_rn(acc[6], acc[7]); w.w = *reinterpret_cast<uint32_t*>(&h);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off) = w;
    }
  }
}

// The upstream gradient of the mean loss and the sum it is the mean of, from
// the device's own count: dloss[n] = 1 / n_valid at counted rows and 0
// elsewhere (all 0 when nothing is counted), and loss_sum[0] = sum_n loss[n]
// (fp64, one block, fixed order). n_valid may be a sum over several ranks' rows.
constexpr int kMeanThreads = 512;
__global__ void __launch_bounds__(kMeanThreads)
    kd_mean_grad_kernel(const float* __restrict__ loss, const uint8_t* __restrict__ mask, int64_t N,
                        const int64_t* __restrict__ n_valid, float* __restrict__ dloss,
                        double* __restrict__ loss_sum) {
  __shared__ double s_part[kMeanThreads];
  const int64_t nv = *n_valid;
  const float g = nv > 0 ? 1.0f / static_cast<float>(nv) : 0.0f;  // fp32, as torch's mask / n_valid
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < N; i += kMeanThreads) {
    const bool counted = (mask == nullptr) || (mask[i] != 0);
    if (dloss) dloss[i] = counted ? g : 0.0f;
    if (loss) acc += static_cast<double>(loss[i]);
  }
  s_part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = kMeanThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s_part[threadIdx.x] += s_part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0 && loss_sum) *loss_sum = s_part[0];
}

// dst[c][r] = src[r][c] for r < R, c < C (bf16 as uint16_t; C a multiple of 8,
// row strides lds / ldd elements, 16-byte aligned rows). One 64 x 64 tile per
// block: 16-byte loads along the source rows into shared memory, 16-byte stores
// along the destination rows. Source rows past R are not read and the
// destination columns for them are not written.
constexpr int kTrTile = 64;
constexpr int kTrPitch = kTrTile + 2;  // 33 words a row: column reads spread over the banks

__global__ void __launch_bounds__(256)
    kd_transpose_kernel(const uint16_t* __restrict__ src, int64_t R, int C, int64_t lds,
                        uint16_t* __restrict__ dst, int64_t ldd) {
  __shared__ uint16_t tile[kTrTile][kTrPitch];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTrTile;
  const int c0 = blockIdx.y * kTrTile;
  const int t = threadIdx.x;
  const int seg = t & 7;  // 8 elements (16 bytes) each
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int rr = (t >> 3) + 32 * pass;
    const int64_t r = r0 + rr;
    const int c = c0 + seg * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < R && c < C) v = *reinterpret_cast<const uint4*>(src + r * lds + c);
    uint32_t* row = reinterpret_cast<uint32_t*>(&tile[rr][seg * 8]);  // 4-byte aligned
    row[0] = v.x;
    row[1] = v.y;
    row[2] = v.z;
    row[3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int cc = (t >> 3) + 32 * pass;  // destination row within the tile
    const int c = c0 + cc;
    const int64_t r = r0 + seg * 8;
    if (c >= C || r >= R) continue;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = static_cast<uint32_t>(tile[seg * 8 + 2 * i][cc]) |
             (static_cast<uint32_t>(tile[seg * 8 + 2 * i + 1][cc]) << 16);
    uint16_t* out = dst + static_cast<int64_t>(c) * ldd + r;
    if (r + 8 <= R) {
      *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int i = 0; i < 8 && r + i < R; ++i)
        out[i] = static_cast<uint16_t>((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
    }
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
