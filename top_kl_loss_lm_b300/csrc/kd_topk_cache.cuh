// kd_topk_cache.cuh — exact per-row top-K of fp32 logits: the selection half of
// the teacher's top-K cache (the logits come from the tcgen05 GEMM, one chunk of
// rows at a time).
//
// One CTA per row (persistent over the chunk's rows). The K-th largest value is
// found exactly by a three-level radix select on an order-preserving 32-bit key
// (11, 11 and 10 bits): each level histograms, in shared memory, the keys whose
// higher bits match the prefix found so far and picks the bin that holds the
// K-th largest. A last pass collects every element above that key and, of those
// equal to it, the ones with the smallest ids (a radix select on the ids when
// more are tied than needed), and a bitonic sort orders the K of them
// (descending logit, then ascending id): the result is deterministic.
//
// The row is normally read once. A sample of the row (runs of 8 consecutive
// logits, one logit in 64 or fewer so that it fits in shared memory) is selected
// first, in shared memory, to a key tau0 that about K + 8 sample strides' worth
// of logits exceed; one pass over the row copies every logit at or above tau0
// (a few hundred) to shared memory, and the exact radix select and the sort
// then run there. If that set holds fewer than K logits or more than
// kSelectCand (heavily tied logits), the row is selected directly: the first
// radix level reads the row, keeps the logits at or above its chosen bin in
// shared memory when they fit, and otherwise every level reads the row again.
#pragma once

#include <cstdint>

namespace kd {

constexpr int kSelectThreads = 512;
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kSelectBins = 2048;
constexpr int kSelectMaxK = 256;
constexpr int kSelectCand = 3072;  // candidates kept in shared memory
constexpr int kSampleStride = 64;  // the threshold sample takes at most every 64th logit
// The bin search gives each thread four consecutive bins: all bins must be owned.
static_assert(4 * kSelectThreads >= kSelectBins, "every histogram bin needs an owning thread");
static_assert(kSelectThreads >= 32 * kSelectWarps && kSelectMaxK <= kSelectCand, "select shape");

// Larger float -> larger key (sign flipped for positives, all bits for negatives).
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Add 1 to hist[bin] for every active lane, one shared atomic per distinct bin.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t live = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(live, bin);
  if ((__ffs(peers) - 1) == static_cast<int>(threadIdx.x & 31)) atomicAdd(&hist[bin], __popc(peers));
}

__global__ void __launch_bounds__(kSelectThreads, 3)
    kd_topk_select_kernel(const float* __restrict__ Z, int64_t ldz, int64_t rows, int V, int K,
                          int32_t* __restrict__ out_idx, float* __restrict__ out_val,
                          const int* __restrict__ run_if) {
  if (run_if != nullptr && *run_if == 0) return;  // a fallback launch that is not needed
  __shared__ uint32_t hist[kSelectBins];
  __shared__ uint32_t warp_sum[kSelectWarps];
  __shared__ uint32_t s_bin, s_above;
  __shared__ uint32_t n_gt, n_eq, n_cand;
  __shared__ uint32_t ckey[kSelectMaxK];
  __shared__ int32_t cidx[kSelectMaxK];
  __shared__ uint32_t cand_key[kSelectCand];
  __shared__ int32_t cand_idx[kSelectCand];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nvec = V / 4;  // float4 part of the row; the tail (V % 4) is read singly

  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* z = Z + row * ldz;
    bool in_smem = false;  // the candidates are in cand_key / cand_idx

    // Calls fn(key, id, valid) for every element of the source with warp-uniform
    // trip counts (fn may use warp-collective operations).
    auto for_each = [&](auto&& fn) {
      if (in_smem) {
        const int n = static_cast<int>(n_cand);
        for (int base = warp * 32; base < n; base += kSelectThreads) {
          const int i = base + lane;
          const bool ok = i < n;
          fn(ok ? cand_key[i] : 0u, ok ? cand_idx[i] : 0, ok);
        }
        return;
      }
      // four 16-byte loads in flight per thread before any of them is used
      constexpr int kUnroll = 4;
      for (int base = warp * 32; base < nvec; base += kUnroll * kSelectThreads) {
        float4 q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v4 = base + u * kSelectThreads + lane;
          q[u] = v4 < nvec ? __ldg(reinterpret_cast<const float4*>(z) + v4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v4 = base + u * kSelectThreads + lane;
          const bool ok = v4 < nvec;
          fn(float_key(q[u].x), 4 * v4 + 0, ok);
          fn(float_key(q[u].y), 4 * v4 + 1, ok);
          fn(float_key(q[u].z), 4 * v4 + 2, ok);
          fn(float_key(q[u].w), 4 * v4 + 3, ok);
        }
      }
      if (warp == 0)
        for (int j = 4 * nvec + lane; j - lane < V; j += 32) {
          const bool ok = j < V;
          fn(float_key(ok ? z[j] : 0.0f), j, ok);
        }
    };

    // Exact radix select over the current source: on return `prefix` is the key of
    // the need0-th largest, `need` the number of elements equal to it to take and
    // eq_last how many elements carry that key. With by_id the keys are ~id of the
    // elements whose logit key equals tau_sel, so the need0-th largest of them
    // marks the need0-th smallest id among logits tied at tau_sel.
    uint32_t prefix = 0;   // key bits fixed so far
    uint32_t need = K;     // elements still to take at or below the prefix
    uint32_t eq_last = 0;  // elements whose whole key equals the result
    int fixed = 0;         // number of fixed high bits
    auto radix_select = [&](uint32_t need0, bool may_shortcut, bool by_id, uint32_t tau_sel) {
    prefix = 0;
    need = need0;
    fixed = 0;
    for (int level = 0; level < 3; ++level) {
      const int bits = level < 2 ? 11 : 10;
      const int shift = 32 - fixed - bits;
      for (int b = tid; b < kSelectBins; b += kSelectThreads) hist[b] = 0;
      if (tid == 0) {  // always a valid bin, even if no thread were to claim one
        s_bin = 0;
        s_above = 0;
      }
      __syncthreads();
      for_each([&](uint32_t k, int id, bool ok) {
        const uint32_t key = by_id ? ~static_cast<uint32_t>(id) : k;
        const bool match = ok && (!by_id || k == tau_sel) &&
                           (fixed == 0 || (key >> (32 - fixed)) == prefix);
        hist_add(hist, (key >> shift) & ((1u << bits) - 1u), match);
      });
      __syncthreads();
      // find the bin holding the need-th largest: thread t owns bins 4t .. 4t+3
      const int nb = 1 << bits;
      uint32_t mine = 0;
      if (4 * tid < nb)
        mine = hist[4 * tid] + hist[4 * tid + 1] + hist[4 * tid + 2] + hist[4 * tid + 3];
      uint32_t incl = mine;  // suffix sum over this warp's lanes (higher lane = higher bins)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      if (lane == 0) warp_sum[warp] = incl;
      __syncthreads();
      uint32_t above_warp = 0;
      for (int w = warp + 1; w < kSelectWarps; ++w) above_warp += warp_sum[w];
      const uint32_t above = above_warp + (incl - mine);  // bins owned by higher threads
      if (4 * tid < nb && above < need && need <= above + mine) {
        uint32_t acc = above;
        for (int b = 4 * tid + 3; b >= 4 * tid; --b) {
          if (acc + hist[b] >= need) {
            s_bin = static_cast<uint32_t>(b);
            s_above = acc;
            break;
          }
          acc += hist[b];
        }
      }
      __syncthreads();
      const uint32_t bin = s_bin, above_bin = s_above;
      const uint32_t in_bin = hist[bin];
      __syncthreads();
      if (level == 2) eq_last = in_bin;
      if (may_shortcut && !by_id && level == 0 &&
          above_bin + in_bin <= static_cast<uint32_t>(kSelectCand)) {
        // everything at or above the chosen top bin fits in shared memory: keep it
        if (tid == 0) n_cand = 0;
        __syncthreads();
        for_each([&](uint32_t k, int id, bool ok) {
          if (ok && (k >> shift) >= bin) {
            const uint32_t slot = atomicAdd(&n_cand, 1u);
            cand_key[slot] = k;
            cand_idx[slot] = id;
          }
        });
        __syncthreads();
        in_smem = true;
      }
      prefix = (prefix << bits) | bin;
      need -= above_bin;
      fixed += bits;
    }
    };

    // 1. threshold from a sample: every kSampleStride-th logit, selected in shared memory
    // the sample is runs of 8 consecutive logits (one 32-byte sector each), one run
    // every 8 * stride logits; positions past V get the smallest key
    const int stride = max(kSampleStride, (V + kSelectCand - 1) / kSelectCand);
    const int runs = (V + 8 * stride - 1) / (8 * stride);
    const int S = 8 * runs;  // <= kSelectCand
    const uint32_t r = min(static_cast<uint32_t>(S),
                           static_cast<uint32_t>((static_cast<int64_t>(K) * S + V - 1) / V) + 8u);
    for (int i = tid; i < S; i += kSelectThreads) {
      const int j = (i >> 3) * (8 * stride) + (i & 7);
      cand_key[i] = j < V ? float_key(__ldg(z + j)) : 0u;
      cand_idx[i] = j;
    }
    if (tid == 0) n_cand = static_cast<uint32_t>(S);
    __syncthreads();
    in_smem = true;
    radix_select(r, false, false, 0u);
    const uint32_t tau0 = prefix;
    __syncthreads();
    // 2. one pass over the row keeps every logit at or above tau0
    if (tid == 0) n_cand = 0;
    __syncthreads();
    in_smem = false;
    for_each([&](uint32_t k, int id, bool ok) {
      if (ok && k >= tau0) {
        const uint32_t slot = atomicAdd(&n_cand, 1u);
        if (slot < static_cast<uint32_t>(kSelectCand)) {
          cand_key[slot] = k;
          cand_idx[slot] = id;
        }
      }
    });
    __syncthreads();
    const uint32_t kept = n_cand;
    __syncthreads();
    if (kept >= static_cast<uint32_t>(K) && kept <= static_cast<uint32_t>(kSelectCand)) {
      in_smem = true;          // the top K are among the kept logits
      radix_select(K, false, false, 0u);
    } else {
      radix_select(K, true, false, 0u);   // select from the row itself
    }
    // prefix is now the exact key of the K-th largest; K - need keys are above it
    const uint32_t tau = prefix;
    const uint32_t take_eq = need;
    const uint32_t n_above = static_cast<uint32_t>(K) - take_eq;
    // more logits tied at tau than needed: take the ones with the smallest ids, so
    // the result does not depend on thread timing
    uint32_t id_cut = 0;  // take tied logits whose ~id >= id_cut
    if (eq_last > take_eq) {
      radix_select(take_eq, false, true, tau);
      id_cut = prefix;
    }
    if (tid == 0) {
      n_gt = 0;
      n_eq = 0;
    }
    __syncthreads();
    for_each([&](uint32_t k, int id, bool ok) {
      if (!ok) return;
      if (k > tau) {
        const uint32_t slot = atomicAdd(&n_gt, 1u);
        if (kd_check(slot < n_above)) {  // exactly n_above keys lie above tau
          ckey[slot] = k;
          cidx[slot] = id;
        }
      } else if (k == tau && ~static_cast<uint32_t>(id) >= id_cut) {
        const uint32_t e = atomicAdd(&n_eq, 1u);
        if (e < take_eq) {  // exactly take_eq qualify; the guard only bounds the slots
          ckey[n_above + e] = k;
          cidx[n_above + e] = id;
        }
      }
    });
    __syncthreads();
    // bitonic sort of the K entries (padded to a power of two) by (key desc, id asc)
    int P = 1;
    while (P < K) P <<= 1;
    for (int i = K + tid; i < P; i += kSelectThreads) {
      ckey[i] = 0u;
      cidx[i] = 0x7FFFFFFF;
    }
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < P; i += kSelectThreads) {
          const int partner = i ^ stride;
          if (partner > i) {
            const bool desc = (i & size) == 0;  // blocks alternate; the final pass is descending
            const uint32_t ka = ckey[i], kb = ckey[partner];
            const int ia = cidx[i], ib = cidx[partner];
            // "a before b" in the final order: larger key, then smaller id
            const bool a_first = (ka > kb) || (ka == kb && ia < ib);
            if (a_first != desc) {
              ckey[i] = kb;
              ckey[partner] = ka;
              cidx[i] = ib;
              cidx[partner] = ia;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < K; i += kSelectThreads) {
      out_idx[row * K + i] = cidx[i];
      out_val[row * K + i] = key_float(ckey[i]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ candidates from the GEMM
//
// The fused form of the cache (no chunk of logits written to memory): a strided
// sample of W's rows gives each row a threshold (the r-th largest sampled logit,
// r a little above K times the sampling rate), the full GEMM's epilogue keeps
// every logit at or above it (kEpiCand), and kd_cand_select_kernel picks the K
// largest of those. A row that kept fewer than K logits, or more than the list
// holds, raises a flag that runs the materialising path for the chunk instead.

// dst[i][:] = src[i * stride][:] for i < rows_out (bf16, D a multiple of 8).
__global__ void __launch_bounds__(256)
    kd_gather_rows_kernel(const uint16_t* __restrict__ src, int64_t stride, int64_t rows_out, int D,
                          uint16_t* __restrict__ dst) {
  const int64_t per_row = D / 8;
  const int64_t n = rows_out * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, c = i - r * per_row;
    reinterpret_cast<uint4*>(dst + r * D)[c] = __ldg(reinterpret_cast<const uint4*>(src + r * stride * D) + c);
  }
}

constexpr int kCandCap = 2048;        // candidates kept per row
constexpr int kCandThreads = 256;

constexpr int kCandBins = 1024;       // histogram bins over a row's key range
constexpr int kCandSel = 512;         // keys kept for the final sort

// Bitonic sort, descending, of keys[0 .. P) in shared memory (P a power of two).
__device__ __forceinline__ void bitonic_desc(unsigned long long* keys, int P, int tid) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += kCandThreads) {
        const int partner = i ^ stride;
        if (partner > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = keys[i], b = keys[partner];
          if ((a > b) != desc && a != b) {
            keys[i] = b;
            keys[partner] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// One CTA per row (grid-stride). The row's candidates become 64-bit keys (logit
// key high, ~id low: distinct, and their descending order is the cache's order,
// ties at equal logits going to the smaller id). Only the K largest are needed:
// a histogram of the logit keys over the row's key range finds the bin that
// holds the K-th largest, the keys in it and above it (K plus that bin's share,
// a few on typical rows) are gathered and sorted, and the first K written out. A
// row where more than kCandSel keys share that bin and those above (heavy ties)
// sorts all its candidates instead. A row with fewer than K or more than cap
// candidates sets *fail.
__global__ void __launch_bounds__(kCandThreads)
    kd_cand_select_kernel(const float* __restrict__ cand_val, const int32_t* __restrict__ cand_id,
                          const int* __restrict__ cand_cnt, int cap, int64_t rows, int K,
                          int32_t* __restrict__ out_idx, float* __restrict__ out_val,
                          int* __restrict__ fail) {
  __shared__ unsigned long long keys[kCandCap];
  __shared__ unsigned long long sel[kCandSel];
  __shared__ int hist[kCandBins];
  __shared__ uint32_t s_lo, s_hi;
  __shared__ int s_bin, s_nsel, s_warp[kCandThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kCandBins / kCandThreads;  // bins a thread scans
  static_assert(kCandBins % kCandThreads == 0, "every bin has one scanning thread");
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const int cnt = cand_cnt[row];
    if (cnt < K || cnt > cap) {
      if (tid == 0) atomicExch(fail, 1);
      continue;  // uniform across the block
    }
    if (tid == 0) {
      s_lo = 0xFFFFFFFFu;
      s_hi = 0u;
      s_nsel = 0;
      s_bin = 0;  // (every key) if no thread claimed a bin, which cnt >= K rules out
    }
    for (int i = tid; i < kCandBins; i += kCandThreads) hist[i] = 0;
    __syncthreads();
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int i = tid; i < cnt; i += kCandThreads) {
      const int64_t o = row * cap + i;
      const uint32_t hk = float_key(cand_val[o]);
      keys[i] = (static_cast<unsigned long long>(hk) << 32) |
                static_cast<unsigned long long>(~static_cast<uint32_t>(cand_id[o]));
      lo = min(lo, hk);
      hi = max(hi, hk);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    if (lane == 0) {
      atomicMin(&s_lo, lo);
      atomicMax(&s_hi, hi);
    }
    __syncthreads();
    const uint32_t klo = s_lo;
    int shift = 0;
    while (((s_hi - klo) >> shift) >= static_cast<uint32_t>(kCandBins)) ++shift;
    for (int i = tid; i < cnt; i += kCandThreads)
      atomicAdd(&hist[(static_cast<uint32_t>(keys[i] >> 32) - klo) >> shift], 1);
    __syncthreads();
    // the bin b holding the K-th largest key: the highest b whose count together
    // with the bins above it reaches K (suffix sums, high bins first)
    int local = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) local += hist[tid * kPer + j];
    int suf = local;  // sum over this lane and the lanes above it in the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_down_sync(0xffffffffu, suf, off);
      if (lane + off < 32) suf += n;
    }
    if (lane == 0) s_warp[warp] = suf;
    __syncthreads();
    int above = suf - local;  // keys in the bins of higher threads
    for (int w = warp + 1; w < kCandThreads / 32; ++w) above += s_warp[w];
    if (above < K && above + local >= K) {
#pragma unroll
      for (int j = kPer - 1; j >= 0; --j) {
        const int h = hist[tid * kPer + j];
        if (above < K && above + h >= K) s_bin = tid * kPer + j;
        above += h;
      }
    }
    __syncthreads();
    const uint32_t bmin = static_cast<uint32_t>(s_bin);
    for (int i = tid; i < cnt; i += kCandThreads) {
      const unsigned long long k = keys[i];
      if (((static_cast<uint32_t>(k >> 32) - klo) >> shift) >= bmin) {
        const int slot = atomicAdd(&s_nsel, 1);
        if (slot < kCandSel) sel[slot] = k;
      }
    }
    __syncthreads();
    const int nsel = s_nsel;
    unsigned long long* src = sel;
    if (nsel <= kCandSel) {
      int P = 1;
      while (P < nsel) P <<= 1;
      for (int i = nsel + tid; i < P; i += kCandThreads) sel[i] = 0ull;  // padding sorts last
      __syncthreads();
      bitonic_desc(sel, P, tid);
    } else {
      int P = 1;
      while (P < cnt) P <<= 1;
      for (int i = cnt + tid; i < P; i += kCandThreads) keys[i] = 0ull;
      __syncthreads();
      bitonic_desc(keys, P, tid);
      src = keys;
    }
    for (int i = tid; i < K; i += kCandThreads) {
      const unsigned long long k = src[i];
      out_idx[row * K + i] = static_cast<int32_t>(~static_cast<uint32_t>(k & 0xFFFFFFFFull));
      out_val[row * K + i] = key_float(static_cast<uint32_t>(k >> 32));
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ row thresholds
//
// thr[row] = the r-th largest of Z[row][0 .. n) (r <= 64), one warp per row and no
// shared memory: the warp holds the 64 largest values seen so far in descending
// order, position p in register p / 32 of lane p % 32. A batch of 32 new values
// (one per lane) is skipped unless one of them beats the current 64th largest;
// otherwise the batch is sorted (bitonic, across lanes) and merged: the element-
// wise max of the list and the reversed batch holds the 64 largest of the union
// as a bitonic sequence, which six compare-exchange stages sort again.
constexpr int kThrMaxRank = 64;
constexpr int kThrWarps = 8;

__device__ __forceinline__ float cmpx_desc(float v, int lane, int stride, bool desc_block) {
  // compare-exchange with lane ^ stride: the lower lane of the pair keeps the
  // larger value when the block is descending
  const float o = __shfl_xor_sync(0xffffffffu, v, stride);
  const bool lower = (lane & stride) == 0;
  return (lower == desc_block) ? fmaxf(v, o) : fminf(v, o);
}

// ONE_LIST (r <= 32): only the 32 largest are kept, one register per lane. A
// batch is skipped unless a value in it beats the current r-th largest (nothing
// below that can reach the final r-th place), which on a random row lets about
// half the batches through compared with testing against the 64th.
template <bool ONE_LIST>
__global__ void __launch_bounds__(kThrWarps * 32)
    kd_row_threshold_kernel(const float* __restrict__ Z, int64_t ldz, int64_t rows, int n, int r,
                            float* __restrict__ thr) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kThrWarps + (threadIdx.x >> 5);
  const int64_t wstep = static_cast<int64_t>(gridDim.x) * kThrWarps;
  const int p = r - 1;
  for (int64_t row = warp0; row < rows; row += wstep) {
    const float* z = Z + row * ldz;
    float a0 = -INFINITY, a1 = -INFINITY;  // positions lane and 32 + lane
    constexpr int kAhead = 8;              // batches loaded before the first is used
    for (int base0 = 0; base0 < n; base0 += 32 * kAhead) {
      float xs[kAhead];
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        const int j = base0 + 32 * u + lane;
        xs[u] = j < n ? __ldg(z + j) : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        float x = xs[u];
        const float rth = __shfl_sync(0xffffffffu, (ONE_LIST || p < 32) ? a0 : a1, p & 31);
        if (__ballot_sync(0xffffffffu, x > rth) == 0u) continue;
        // sort the batch descending across the lanes
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1) {
          const bool desc_block = (lane & size) == 0 || size == 32;
#pragma unroll
          for (int stride = size >> 1; stride > 0; stride >>= 1) x = cmpx_desc(x, lane, stride, desc_block);
        }
        if constexpr (ONE_LIST) {
          // the 32 largest of the list and the batch, reversed: a bitonic sequence
          a0 = fmaxf(a0, __shfl_sync(0xffffffffu, x, 31 - lane));
#pragma unroll
          for (int stride = 16; stride > 0; stride >>= 1) a0 = cmpx_desc(a0, lane, stride, true);
        } else {
          // positions 32..63 against the batch reversed (positions 0..31 keep theirs:
          // the padded half of the batch is -inf there)
          a1 = fmaxf(a1, __shfl_sync(0xffffffffu, x, 31 - lane));
          // bitonic sequence of 64 -> descending: stride 32 inside the lane, then 16..1
          const float hi = fmaxf(a0, a1), lo = fminf(a0, a1);
          a0 = hi;
          a1 = lo;
#pragma unroll
          for (int stride = 16; stride > 0; stride >>= 1) {
            a0 = cmpx_desc(a0, lane, stride, true);
            a1 = cmpx_desc(a1, lane, stride, true);
          }
        }
      }
    }
    const float t = __shfl_sync(0xffffffffu, (ONE_LIST || p < 32) ? a0 : a1, p & 31);
    if (lane == 0) thr[row] = t;
  }
}

}  // namespace kd
