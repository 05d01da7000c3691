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
// Warp 0 is the copy engine's driver: it keeps NBUF row buffers in a ring (the
// library uses two), loading the next row while this one is reduced and
// storing each finished dZ row; warps 1..8 compute. Two such CTAs share an SM
// when the slices are small enough, so each SM runs two row pipelines. Partials travel to every CTA of the cluster with st.async onto an
// mbarrier, so no cluster-wide barrier sits in the row loop and the copies
// never wait on the arithmetic. Every wait is bounded: a CTA that gives up
// records KD_ERR_TIMEOUT, skips the remaining work, and its peers' waits for
// its partials run out in turn.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_bf16.h>

#include "kd_ptx.cuh"

namespace kd {

constexpr int kLogitsThreads = 256;  // compute threads (warps 1..8) with the gradient
constexpr int kLogitsThreadsLossOnly = 128;  // loss only: lighter CTAs, four per SM
constexpr int kLogitsMaxWarps = kLogitsThreads / 32;
constexpr int kLogitsMaxCluster = 8;
constexpr int kLogitsMaxBuffers = 4;
constexpr int kLogitsMaxK = 256;  // teacher entries per row (two per compute thread at most)
static_assert(kLogitsMaxK <= 2 * kLogitsThreadsLossOnly, "a compute thread holds at most two entries");

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

// Shared memory of one CTA: NBUF row slices, then the small parts.
__host__ __device__ constexpr size_t logits_smem_bytes(int Vs, int nbuf) {
  return static_cast<size_t>(nbuf) * Vs * 2      // row slices (bf16)
         + 2 * kLogitsMaxCluster * 16            // cluster partials, two parities
         + 2 * kLogitsMaxWarps * 16              // block reduction scratch, two parities
         + 2 * kLogitsMaxK * 8                   // the row's teacher entries, two parities
         + (2 * kLogitsMaxBuffers + 2) * 8 + 16; // full / empty / exchange barriers, abort flag
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

// Barrier among the NT compute threads only (named barrier 1).
template <int NT>
__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// CL: CTAs per row (cluster size); NBUF: row buffers per CTA; NT: compute threads.
template <int CL, int NBUF, int NT>
__global__ void __launch_bounds__(NT + 32, NT <= 128 ? 4 : 2) kd_logits_kernel(const LogitsArgs a) {
  constexpr int kLogitsWarps = NT / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const size_t slice_bytes = static_cast<size_t>(a.Vs) * 2;
  auto buf = [&](int b) { return reinterpret_cast<uint16_t*>(smem + b * slice_bytes); };
  float4* exch = reinterpret_cast<float4*>(smem + NBUF * slice_bytes);  // [2][kLogitsMaxCluster]
  float4* red = exch + 2 * kLogitsMaxCluster;                          // [2][max warps]
  int2* spairs = reinterpret_cast<int2*>(red + 2 * kLogitsMaxWarps);    // [2][max K]
  uint64_t* full = reinterpret_cast<uint64_t*>(spairs + 2 * kLogitsMaxK);
  uint64_t* empty = full + kLogitsMaxBuffers;
  uint64_t* xbar = empty + kLogitsMaxBuffers;                          // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(xbar + 2);

  const int tid = threadIdx.x;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t cluster = blockIdx.x / CL;
  const int64_t nclusters = gridDim.x / CL;
  const int lo = static_cast<int>(rank) * a.Vs;
  const int len = max(0, min(a.V, lo + a.Vs) - lo);  // columns of this slice (multiple of 8)
  const uint32_t bytes = static_cast<uint32_t>(len) * 2u;
  const int64_t rows = cluster < a.N ? (a.N - cluster + nclusters - 1) / nclusters : 0;
  const bool grad = a.dZ != nullptr;

  if (tid == 0) {
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kLogitsWarps);
    }
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if constexpr (CL > 1)
    cluster_sync();  // peers' barriers exist before any st.async reaches them
  else
    __syncthreads();

  if (tid < 32) {
    // ---------------------------------------------------------------- copy driver
    if (tid == 0) {
      auto store = [&](int64_t j, int b) {
        if (grad && bytes && !*abort_flag) {
          bulk_store_1d(a.dZ + (cluster + j * nclusters) * a.lddz + lo, buf(b), bytes);
          bulk_commit_group();
        }
      };
      for (int64_t j = 0; j < rows; ++j) {
        const int b = static_cast<int>(j % NBUF);
        const int64_t u = j / NBUF;
        if (u > 0) {
          // row j - NBUF is finished in this buffer: store its dZ, let the store
          // read the buffer, then reuse it
          if (!mbar_wait_bounded(&empty[b], static_cast<uint32_t>((u - 1) & 1), abort_flag,
                                 a.timeout_ns, a.status, 6))
            break;
          store(j - NBUF, b);
          bulk_wait_group_read<0>();
        }
        mbar_arrive_expect_tx(&full[b], bytes);
        if (bytes) bulk_load_1d(buf(b), a.Z + (cluster + j * nclusters) * a.ldz + lo, bytes, &full[b]);
      }
      for (int64_t j = rows > NBUF ? rows - NBUF : 0; j < rows && !*abort_flag; ++j) {
        const int b = static_cast<int>(j % NBUF);
        if (!mbar_wait_bounded(&empty[b], static_cast<uint32_t>((j / NBUF) & 1), abort_flag,
                               a.timeout_ns, a.status, 6))
          break;
        store(j, b);
      }
      bulk_wait_group_all();
    }
    __syncwarp();  // the warp reconverges before the final cluster barrier
  } else {
    // ---------------------------------------------------------------- compute warps
    const int ctid = tid - 32;
    const int cwarp = ctid >> 5, lane = ctid & 31;
    const int nvec = len / 8;
    const int K = a.K;
    for (int64_t j = 0; j < rows; ++j) {
      const int64_t row = cluster + j * nclusters;
      const int b = static_cast<int>(j % NBUF);
      const int par = static_cast<int>(j & 1);
      // The row's teacher entries and per-row values are read from global memory
      // here and used only after pass 1's vector loop, so their latency hides
      // behind it; the entries also go to shared memory for pass 2.
      int2 q0 = make_int2(INT_MAX, 0), q1 = make_int2(INT_MAX, 0);
      if (ctid < K) q0 = __ldg(&a.pairs[row * K + ctid]);
      if (ctid + NT < K) q1 = __ldg(&a.pairs[row * K + ctid + NT]);
      const bool counted = (a.mask == nullptr) || (a.mask[row] != 0);
      const float dl = grad ? __ldg(&a.dloss[row]) : 0.0f;
      const float entr = (rank == 0 && ctid == 0) ? __ldg(&a.ent[row]) : 0.0f;
      int2* sp = spairs + par * kLogitsMaxK;
      bool work = !*abort_flag &&
                  mbar_wait_bounded(&full[b], static_cast<uint32_t>((j / NBUF) & 1), abort_flag,
                                    a.timeout_ns, a.status, 6);
      const uint16_t* zrow = buf(b);

      // ---- pass 1: online max / sum of exponentials, and the teacher's cross term
      // running (max, sum of exponentials) in base 2; the sum in two lanes, packed
      float msx = -INFINITY;
      uint64_t msy2 = f32x2(0.0f, 0.0f);
      float cross = 0.0f;
      int2 pr = make_int2(INT_MAX, 0);
      float zk = 0.0f;
      bool mine = false;  // this thread's teacher entry falls in the slice
      if (work) {
        for (int v = ctid; v < nvec; v += NT) {
          const uint4 w = *reinterpret_cast<const uint4*>(zrow + 8 * v);
          const float z[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                              bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
          float mx = z[0];
#pragma unroll
          for (int i = 1; i < 8; ++i) mx = fmaxf(mx, z[i]);
          const float mnew = fmaxf(msx, mx * a.scale2);
          // the eight arguments z*log2e/T - max as four packed FMAs, the sum as
          // packed adds (the exponentials stay one MUFU instruction each)
          const uint64_t s2 = f32x2(a.scale2, a.scale2), nm2 = f32x2(-mnew, -mnew);
          const uint64_t e0 = ex2_f32x2(fma_f32x2(f32x2(z[0], z[1]), s2, nm2));
          const uint64_t e1 = ex2_f32x2(fma_f32x2(f32x2(z[2], z[3]), s2, nm2));
          const uint64_t e2 = ex2_f32x2(fma_f32x2(f32x2(z[4], z[5]), s2, nm2));
          const uint64_t e3 = ex2_f32x2(fma_f32x2(f32x2(z[6], z[7]), s2, nm2));
          const float c = ex2_approx(msx - mnew);
          msy2 = fma_f32x2(msy2, f32x2(c, c), add_f32x2(add_f32x2(e0, e1), add_f32x2(e2, e3)));
          msx = mnew;
        }
        // teacher entries ctid and ctid + NT; the first one is kept for the
        // gradient's correction (with the gradient NT >= K, so that is every entry)
        if (ctid < K) {
          sp[ctid] = q0;
          if (q0.x >= lo && q0.x < lo + len) {
            const float zq = __uint_as_float(static_cast<uint32_t>(zrow[q0.x - lo]) << 16);
            cross += __int_as_float(q0.y) * zq;
            pr = q0;
            zk = zq;
            mine = true;
          }
        }
        if (ctid + NT < K) {
          sp[ctid + NT] = q1;
          if (q1.x >= lo && q1.x < lo + len)
            cross += __int_as_float(q1.y) *
                     __uint_as_float(static_cast<uint32_t>(zrow[q1.x - lo]) << 16);
        }
      }
      float2 ms;
      {
        float ylo, yhi;
        f32x2_split(msy2, ylo, yhi);
        ms = make_float2(msx, ylo + yhi);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, ms.x, o),
                                         __shfl_xor_sync(0xffffffffu, ms.y, o));
        ms = merge_ms(ms, other);
        cross += __shfl_xor_sync(0xffffffffu, cross, o);
      }
      float4* rd = red + par * kLogitsWarps;
      if (lane == 0) rd[cwarp] = make_float4(ms.x, ms.y, cross, 0.0f);
      compute_sync<NT>();
      float2 rms = make_float2(-INFINITY, 0.0f);
      float rcross = 0.0f;
#pragma unroll
      for (int w = 0; w < kLogitsWarps; ++w) {
        const float4 r = rd[w];
        rms = merge_ms(rms, make_float2(r.x, r.y));
        rcross += r.z;
      }

      // ---- merge over the cluster: every CTA sends its partial to every CTA
      if constexpr (CL > 1) {
        float4* slot = exch + par * kLogitsMaxCluster;
        if (ctid == 0) mbar_arrive_expect_tx(&xbar[par], CL * 16);
        if (ctid < CL) {
          const uint32_t dst = mapa_shared(smem_u32(&slot[rank]), static_cast<uint32_t>(ctid));
          const uint32_t bar = mapa_shared(smem_u32(&xbar[par]), static_cast<uint32_t>(ctid));
          st_async_v4(dst, make_float4(rms.x, rms.y, rcross, 0.0f), bar);
        }
        work = mbar_wait_bounded(&xbar[par], static_cast<uint32_t>((j >> 1) & 1), abort_flag,
                                 a.timeout_ns, a.status, 6) && work;
        rms = make_float2(-INFINITY, 0.0f);
        rcross = 0.0f;
#pragma unroll
        for (int r = 0; r < CL; ++r) {
          const float4 q = slot[r];
          rms = merge_ms(rms, make_float2(q.x, q.y));
          rcross += q.z;
        }
      }
      const float lse2 = rms.x + log2f(rms.y);
      if (rank == 0 && ctid == 0 && work) {
        const double lse = static_cast<double>(lse2) * 0.6931471805599453;
        a.lse[row] = static_cast<float>(lse);
        a.loss[row] = counted ? static_cast<float>(static_cast<double>(entr) -
                                                   static_cast<double>(rcross) * a.inv_T + lse)
                              : 0.0f;
      }

      // ---- pass 2: dZ in place (the copy driver stores it)
      if (grad && work) {
        const float gs = counted ? dl * a.inv_T : 0.0f;
        uint16_t* drow = buf(b);
        for (int v = ctid; v < nvec; v += NT) {
          uint4* p = reinterpret_cast<uint4*>(drow + 8 * v);
          uint4 w = *p;
          if (counted) {
            const float z[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
            const uint64_t s2 = f32x2(a.scale2, a.scale2), nl2 = f32x2(-lse2, -lse2);
            const uint64_t g2 = f32x2(gs, gs);
            float d[8];
#pragma unroll
            for (int i = 0; i < 8; i += 2)
              f32x2_split(mul_f32x2(g2, ex2_f32x2(fma_f32x2(f32x2(z[i], z[i + 1]), s2, nl2))), d[i],
                          d[i + 1]);
            w = make_uint4(f2_to_bf16x2(d[0], d[1]), f2_to_bf16x2(d[2], d[3]),
                           f2_to_bf16x2(d[4], d[5]), f2_to_bf16x2(d[6], d[7]));
          } else {
            w = make_uint4(0u, 0u, 0u, 0u);
          }
          *p = w;
        }
        compute_sync<NT>();  // the vectors are written before single entries are corrected
        if (counted && mine && (ctid == 0 || sp[ctid - 1].x != pr.x)) {
          float P = __int_as_float(pr.y);  // merge a run of repeated ids
          for (int k2 = ctid + 1; k2 < K; ++k2) {
            const int2 q = sp[k2];
            if (q.x != pr.x) break;
            P += __int_as_float(q.y);
          }
          const float d = gs * (ex2_approx(fmaf(zk, a.scale2, -lse2)) - P);
          const __nv_bfloat16 h = __float2bfloat16_rn(d);
          drow[pr.x - lo] = *reinterpret_cast<const uint16_t*>(&h);
        }
        fence_proxy_async_shared();  // the copy engine reads what these threads wrote
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[b]);
    }
  }

  if (*abort_flag) {
    // copies issued before giving up land within microseconds
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if constexpr (CL > 1) cluster_sync();  // no CTA leaves while a peer may still write to it
}

}  // namespace kd
