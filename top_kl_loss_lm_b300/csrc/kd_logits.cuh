// kd_logits.cuh — top-K KL loss and its logit gradient from logits that were
// already computed (the forward-chunked form: the student's logits exist in
// full, the teacher stays sparse, the loss is taken one slice of positions at a
// time).
//
// One cluster of CL CTAs owns one row of the N x V logits at a time; CTA r of the
// cluster holds columns [r*Vs, (r+1)*Vs) of the row in shared memory, loaded
// with one bulk copy. The row is read from HBM once and, when the gradient is
// wanted, dZ is written once, in place in shared memory and then by one bulk
// store: 4 bytes of HBM traffic per logit, the least the operation allows.
//
//   pass 1   per-thread online (max, sum of 2^(z*log2e/T - max)), merged over the
//            block and then over the cluster through distributed shared memory;
//            the teacher's cached ids that fall in the slice give sum_k p_k z_k
//   loss     entropy - (sum_k p_k z_k)/T + lse, written by the cluster's CTA 0
//   pass 2   dZ = (g/T)(2^(z*log2e/T - lse2) - P~) for every column, rounded to
//            bf16 in place; the teacher's ids get their exact fp32 value
//            (repeated ids merged) before rounding; then one bulk store
//
// Two row buffers per CTA: the next row's bulk copy runs while this row is
// reduced. Every wait is bounded; a CTA that gives up keeps taking part in the
// cluster barriers (so no peer can wait forever) and only skips work.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_bf16.h>

#include "kd_ptx.cuh"

namespace kd {

constexpr int kLogitsThreads = 256;
constexpr int kLogitsWarps = kLogitsThreads / 32;
constexpr int kLogitsMaxCluster = 8;

struct LogitsArgs {
  const uint16_t* Z;     // N x V bf16 logits, row stride ldz elements
  int64_t ldz;
  uint16_t* dZ;          // N x V bf16 gradient (row stride lddz), or nullptr for the loss only
  int64_t lddz;
  const int2* pairs;     // N x K sorted (id, p bits) from the prep kernel
  const float* ent;      // N teacher entropy sum_j P_j log P_j
  const uint8_t* mask;   // N (nullptr: all rows counted)
  const float* dloss;    // N upstream gradient (used when dZ != nullptr)
  float* loss;
  float* lse;
  int64_t N;
  int V, K, Vs;          // Vs: columns per CTA slice (multiple of 64)
  float scale2;          // log2(e) / T
  float inv_T;
  int* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t logits_smem_bytes(int Vs) {
  return 2 * static_cast<size_t>(Vs) * 2       // two row buffers (bf16)
         + 2 * kLogitsMaxCluster * 16           // cluster exchange slots, two parities
         + kLogitsWarps * 16                    // block reduction scratch
         + 2 * 8 + 16;                          // two mbarriers, abort flag
}

__device__ __forceinline__ float2 merge_ms(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.0f);
  return make_float2(m, a.y * ex2_approx(a.x - m) + b.y * ex2_approx(b.x - m));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t f2_to_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int CL>
__global__ void __launch_bounds__(kLogitsThreads, 1) kd_logits_kernel(const LogitsArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  auto buf = [&](int b) { return reinterpret_cast<uint16_t*>(smem + static_cast<size_t>(b) * a.Vs * 2); };
  float4* exch = reinterpret_cast<float4*>(smem + static_cast<size_t>(a.Vs) * 4);  // [2][CL]
  float4* red = exch + 2 * kLogitsMaxCluster;                                     // [warps]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kLogitsWarps);               // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t cluster = blockIdx.x / CL;
  const int64_t nclusters = gridDim.x / CL;
  const int lo = static_cast<int>(rank) * a.Vs;
  const int len = max(0, min(a.V, lo + a.Vs) - lo);  // columns of this slice (multiple of 8)
  const uint32_t bytes = static_cast<uint32_t>(len) * 2u;
  const int nvec = len / 8;
  const int K = a.K;

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if constexpr (CL > 1)
    cluster_sync();
  else
    __syncthreads();

  auto load_row = [&](int64_t row, int b) {  // thread 0 only
    mbar_arrive_expect_tx(&full[b], bytes);
    if (bytes) bulk_load_1d(buf(b), a.Z + row * a.ldz + lo, bytes, &full[b]);
  };
  if (tid == 0 && cluster < a.N) load_row(cluster, 0);

  int i = 0;
  for (int64_t row = cluster; row < a.N; row += nclusters, ++i) {
    const int b = i & 1;
    const int64_t next = row + nclusters;
    if (tid == 0 && next < a.N && !*abort_flag) {
      if (a.dZ) bulk_wait_group_read<0>();  // the store from the other buffer has read it
      load_row(next, b ^ 1);
    }
    const bool have = mbar_wait_bounded(&full[b], static_cast<uint32_t>((i >> 1) & 1), abort_flag,
                                        a.timeout_ns, a.status, 6);
    const bool work = __syncthreads_and(have ? 1 : 0) != 0;
    const uint16_t* zrow = buf(b);

    // ---- pass 1: online max / sum of exponentials, and the teacher's cross term
    float2 ms = make_float2(-INFINITY, 0.0f);
    float cross = 0.0f;
    int2 pr = make_int2(INT_MAX, 0);
    float zk = 0.0f;
    bool mine = false;  // this thread's teacher entry falls in the slice
    if (work) {
      for (int v = tid; v < nvec; v += kLogitsThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(zrow + 8 * v);
        float z[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                      bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        float mx = z[0];
#pragma unroll
        for (int j = 1; j < 8; ++j) mx = fmaxf(mx, z[j]);
        const float mnew = fmaxf(ms.x, mx * a.scale2);
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += ex2_approx(fmaf(z[j], a.scale2, -mnew));
        ms.y = ms.y * ex2_approx(ms.x - mnew) + s;
        ms.x = mnew;
      }
      if (tid < K) {
        pr = __ldg(&a.pairs[row * K + tid]);
        if (pr.x >= lo && pr.x < lo + len) {
          zk = __uint_as_float(static_cast<uint32_t>(zrow[pr.x - lo]) << 16);
          cross = __int_as_float(pr.y) * zk;
          mine = true;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, ms.x, o),
                                       __shfl_xor_sync(0xffffffffu, ms.y, o));
      ms = merge_ms(ms, other);
      cross += __shfl_xor_sync(0xffffffffu, cross, o);
    }
    if (lane == 0) red[warp] = make_float4(ms.x, ms.y, cross, 0.0f);
    __syncthreads();
    float2 bms = make_float2(-INFINITY, 0.0f);
    float bcross = 0.0f;
#pragma unroll
    for (int w = 0; w < kLogitsWarps; ++w) {
      const float4 r = red[w];
      bms = merge_ms(bms, make_float2(r.x, r.y));
      bcross += r.z;
    }

    // ---- merge over the cluster (distributed shared memory)
    float2 rms = bms;
    float rcross = bcross;
    if constexpr (CL > 1) {
      float4* slot = exch + b * kLogitsMaxCluster;
      if (tid < CL) {
        const uint32_t dst = mapa_shared(smem_u32(&slot[rank]), static_cast<uint32_t>(tid));
        st_cluster_v4(dst, make_float4(bms.x, bms.y, bcross, 0.0f));
      }
      cluster_sync();
      rms = make_float2(-INFINITY, 0.0f);
      rcross = 0.0f;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        const float4 p = slot[r];
        rms = merge_ms(rms, make_float2(p.x, p.y));
        rcross += p.z;
      }
    }
    const float lse2 = rms.x + log2f(rms.y);
    const bool counted = (a.mask == nullptr) || (a.mask[row] != 0);
    if (rank == 0 && tid == 0 && work) {
      const double lse = static_cast<double>(lse2) * 0.6931471805599453;
      a.lse[row] = static_cast<float>(lse);
      a.loss[row] = counted ? static_cast<float>(static_cast<double>(a.ent[row]) -
                                                 static_cast<double>(rcross) * a.inv_T + lse)
                            : 0.0f;
    }

    // ---- pass 2: dZ in place, then one bulk store
    if (a.dZ && work) {
      const float gs = counted ? a.dloss[row] * a.inv_T : 0.0f;
      uint16_t* drow = buf(b);
      for (int v = tid; v < nvec; v += kLogitsThreads) {
        uint4* p = reinterpret_cast<uint4*>(drow + 8 * v);
        uint4 w = *p;
        if (counted) {
          const float z[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                              bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
          float d[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) d[j] = gs * ex2_approx(fmaf(z[j], a.scale2, -lse2));
          w = make_uint4(f2_to_bf16x2(d[0], d[1]), f2_to_bf16x2(d[2], d[3]),
                         f2_to_bf16x2(d[4], d[5]), f2_to_bf16x2(d[6], d[7]));
        } else {
          w = make_uint4(0u, 0u, 0u, 0u);
        }
        *p = w;
      }
      __syncthreads();
      if (counted && mine && (tid == 0 || __ldg(&a.pairs[row * K + tid - 1]).x != pr.x)) {
        float P = __int_as_float(pr.y);  // merge a run of repeated ids
        for (int k2 = tid + 1; k2 < K; ++k2) {
          const int2 q = __ldg(&a.pairs[row * K + k2]);
          if (q.x != pr.x) break;
          P += __int_as_float(q.y);
        }
        const float d = gs * (ex2_approx(fmaf(zk, a.scale2, -lse2)) - P);
        const __nv_bfloat16 h = __float2bfloat16_rn(d);
        drow[pr.x - lo] = *reinterpret_cast<const uint16_t*>(&h);
      }
      fence_proxy_async_shared();
      __syncthreads();
      if (tid == 0 && bytes) {
        bulk_store_1d(a.dZ + row * a.lddz + lo, drow, bytes);
        bulk_commit_group();
      }
    }
    __syncthreads();  // this buffer is free for the row after next
  }

  if (tid == 0) bulk_wait_group_all();
  if (*abort_flag) {
    // copies issued before giving up land within microseconds
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if constexpr (CL > 1) cluster_sync();  // no CTA leaves while a peer may still write to it
}

}  // namespace kd
