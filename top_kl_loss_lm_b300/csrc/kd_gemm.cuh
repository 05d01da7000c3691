// kd_gemm.cuh — persistent, warp-specialised tcgen05 GEMM for sm_103a with the
// loss epilogues fused in.
//
// The loss runs it on CTA pairs (cluster of 2, cta_group::2): a 256 x BN tile per
// pair, each CTA holding 128 rows of A and half of B per k-block; the single-CTA
// form (128 x BN tiles) remains for the GEMM test hook.
//
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) k-blocks (on a
//               pair, both CTAs' copies complete on the first CTA's barrier)
//   warp 1      TMEM owner + MMA issuer (first CTA of a pair): M x BN x 16 bf16
//               MMAs into one of two fp32 TMEM accumulators (2 x 256 columns),
//               so the epilogue of one tile overlaps the main loop of the next
//   warps 2..5  epilogue: each thread owns one accumulator row (TMEM lane) of
//               its CTA
//
// Epilogues:
//   kEpiFwd   online max / sum-of-exp of Z/T over the unit's vocabulary tiles
//             (partial per row and split) + gather of Z at the row's sorted
//             teacher ids that fall in the tile
//   kEpiDz    dZ = (g/T)(exp(Z/T - lse) - P~) with P~ scattered from the sorted
//             ids, rounded to bf16 and stored into the chunk's dZ buffer by TMA
//   kEpiDh    dH tile (bf16, or fp32 partial per k-split)
//   kEpiDw    dW tile, stored or added to the existing fp32 values
//   kEpiPlain fp32 C tile (mainloop test hook, the teacher's logits)
//   kEpiCand  the teacher cache's candidates: every logit at or above its row's
//             threshold is appended (value, id) to the row's candidate list
// fp32 tiles (dW, plain, dH partials) are staged per warp in shared memory as
// 32 x 16 boxes and written by TMA: a bulk-tensor store, or for an accumulating
// dW a bulk-tensor add that L2 applies (one owner per tile, so no atomics race).
//
// Operand layouts in shared memory are the TMA 128-byte-swizzled boxes: a
// K-major operand is rows x 64 bf16 (one 128-byte line per row); an MN-major
// operand is 64-wide MN slabs of 64 k-rows, 8 KB each.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "kd_ptx.cuh"
#include "kd_sched.h"

namespace kd {

// fp32 output boxes staged in shared memory for the TMA store / reduce epilogue:
// 32 rows x 16 columns (64 bytes a row, 64-byte swizzle), two boxes per 32-column
// TMEM chunk, two chunks in flight per epilogue warp.
constexpr int kOutBoxCols = 16;
constexpr int kOutBoxBytes = 32 * kOutBoxCols * 4;       // 2 KB
constexpr int kOutChunkBytes = 2 * kOutBoxBytes;          // 4 KB: one 32-column chunk
constexpr int kStagingBytes = 4 * 2 * kOutChunkBytes;     // 4 warps x 2 chunks = 32 KB

// Per-CTA pipeline geometry. Single CTA: 128 x 256 tiles, 48 KB k-blocks, 4 stages.
// CTA pair (cta_group::2): 256 x BN tiles; each CTA holds 128 rows of A and half
// of B (<= 128 columns) per k-block, 32 KB, 6 stages.
template <bool PAIR>
struct Geo {
  static constexpr int kTileRows = PAIR ? 256 : 128;
  static constexpr int kBRows = PAIR ? 128 : 256;               // B rows (columns of D) per CTA
  static constexpr int kAStageBytes = kBM * kBK * 2;              // 16 KB
  static constexpr int kBStageBytes = kBRows * kBK * 2;           // 16 / 32 KB
  static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kRingBytes + kStagingBytes + 1024 /*align*/ + 256 /*barriers*/;
};
constexpr int kSlabBytes = 64 * kBK * 2;         // one 64-wide MN slab of a k-block: 8 KB
constexpr int kFwdExtraStages = 1;               // ring stages the forward gains from staging
constexpr int kGemmThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kGemmSmemBytes = Geo<false>::kSmemBytes > Geo<true>::kSmemBytes ? Geo<false>::kSmemBytes
                                                                               : Geo<true>::kSmemBytes;

enum Epi : int { kEpiFwd = 0, kEpiDz = 1, kEpiDh = 2, kEpiDw = 3, kEpiPlain = 4, kEpiCand = 5 };

struct GemmArgs {
  Sched sched;
  int M;              // valid output rows (fwd: N, dz/dh: rows in chunk, dw: V, plain: M)
  int Ncols;          // valid output columns (fwd/dz: V, dh/dw: D, plain: N)
  int BN;             // tile width = MMA N (multiple of 16, <= 256)
  uint32_t idesc;
  int a_row_off;      // K-major A: row offset added to the tile row (chunk start in H)
  int b_k_off;        // MN-major B: k-row offset (chunk start in H for dW)
  int64_t row_base;   // global token of local row 0 (fwd, dz, dh)
  int K;              // teacher top-K
  float scale2;       // log2(e) / T
  float inv_T;
  const int2* pairs;  // N x K sorted (id, p bits)
  float* zk;          // N x K gathered logits (sorted order)
  float2* part;       // N x slots (max, sum) in base-2 units
  int slots;
  const float* lse;
  const float* dloss;
  const uint8_t* mask;
  uint16_t* dz;       // chunk dZ buffer, row stride dz_ld
  int64_t dz_ld;
  float* out_f32;     // dh partials / dW / plain C
  int64_t ld_out;
  int64_t part_stride;  // dh: elements per k-split slice
  uint16_t* out_bf16;   // dH
  int accumulate;       // dW: add to existing values
  int out_slot_rows;    // dh partials: rows of one k-split slice in the tmC tensor
  int* status;
  uint64_t timeout_ns;
  int dh_partials;      // dH: fp32 partials through tmC even without a k-split
  // kEpiCand: row r's threshold is thr[r * thr_stride + thr_stride - 1]; its list is
  // cand_val / cand_id [r * cand_cap ...], cand_cnt[r] counts every logit that passed
  const float* thr;
  int thr_stride;
  float* cand_val;
  int32_t* cand_id;
  int* cand_cnt;
  int cand_cap;
  const int* run_if;    // if set and *run_if == 0 the launch does nothing (a fallback)
};

// fp32 tiles leave through tmC (TMA store, or TMA add for an accumulating dW):
// dW, the plain GEMM, and the dH partials (k-split, or an fp32 dH).
template <int EPI>
__host__ __device__ __forceinline__ bool uses_tma_out(const GemmArgs& a) {
  return EPI == kEpiDz || EPI == kEpiDw || EPI == kEpiPlain ||
         (EPI == kEpiDh && (a.sched.KS > 1 || a.dh_partials != 0));
}

// One 32-column TMEM chunk of a warp's 32 rows -> two swizzled 32 x 16 fp32 boxes
// in shared memory -> TMA store or add at (x0, y0). Lane r holds row r. The
// 64-byte swizzle puts 16-byte piece j of row r at piece j ^ ((r >> 1) & 3),
// which is what the tensor map's SWIZZLE_64B expects and keeps the eight
// lanes of each 128-bit store phase on distinct banks.
__device__ __forceinline__ void send_chunk(const CUtensorMap* map, uint8_t* buf, const float (&v)[32],
                                           int lane, int x0, int y0, int boxes, bool add) {
  const uint32_t base = smem_u32(buf) + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t addr = base + b * kOutBoxBytes + ((static_cast<uint32_t>(j) ^ sw) << 4);
      st_shared_v4(addr, v[16 * b + 4 * j + 0], v[16 * b + 4 * j + 1], v[16 * b + 4 * j + 2],
                   v[16 * b + 4 * j + 3]);
    }
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    for (int b = 0; b < boxes; ++b) {
      if (add)
        tma_reduce_add_2d<4>(map, buf + b * kOutBoxBytes, x0 + kOutBoxCols * b, y0);
      else
        tma_store_2d<4>(map, buf + b * kOutBoxBytes, x0 + kOutBoxCols * b, y0);
    }
    bulk_commit_group();
  }
}

// v[j] for a j known only at run time, without indexing the register array (which
// would put it in local memory): a tree of selects on the bits of j.
__device__ __forceinline__ float select32(const float (&v)[32], int j) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (j & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = (j & 2) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (j & 4) ? b[2 * i + 1] : b[2 * i];
#pragma unroll
  for (int i = 0; i < 2; ++i) d[i] = (j & 8) ? c[2 * i + 1] : c[2 * i];
  return (j & 16) ? d[1] : d[0];
}

__device__ __forceinline__ void sub_at32(float (&v)[32], int j, float x) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = (j == i) ? v[i] - x : v[i];
}

__device__ __forceinline__ int lower_bound_id(const int2* p, int K, int target) {
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&p[mid].x) < target)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// bf16 variant for the dZ chunk: 32 rows x 32 columns rounded to bf16 (64 bytes
// a row, same 64-byte swizzle), one TMA store at (x0, y0).
__device__ __forceinline__ void send_chunk_bf16(const CUtensorMap* map, uint8_t* buf,
                                                const float (&v)[32], int lane, int x0, int y0) {
  const uint32_t base = smem_u32(buf) + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t addr = base + ((static_cast<uint32_t>(j) ^ sw) << 4);
    st_shared_v4_b32(addr, pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                     pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d<2>(map, buf, x0, y0);
    bulk_commit_group();
  }
}

// kEpiCand on one accumulator tile of this warp's 32 rows (lane = row). A few
// hundred of a row's ~200K logits reach its threshold, so almost every 32 x 32
// block of a tile holds one, and an atomic per passing logit would put several
// L2 round trips per block on the epilogue's path. So a first pass over the
// tile's TMEM chunks marks each row's passing columns (one bit mask per chunk),
// one atomic per row reserves that many slots of the row's list, and a second
// pass reads the chunks that hold any passing logit again and writes them.
// Columns past the vocabulary's end never pass. cand_cnt counts every passing
// logit, written or not, so a list that overflowed is seen by the select.
__device__ __forceinline__ void cand_tile(uint32_t tacc, int col_tile, float theta, int row,
                                          bool row_ok, const GemmArgs& args) {
  uint32_t mask[kBNMax / 32];
  int total = 0;
#pragma unroll
  for (int c = 0; c < kBNMax / 32; ++c) {
    mask[c] = 0u;
    const int col0 = col_tile + 32 * c;
    if (32 * c < args.BN && col0 < args.Ncols) {  // warp-uniform
      float v[32];
      __syncwarp();
      tmem_ld32(tacc + 32 * c, v);
      uint32_t m = 0u;
#pragma unroll
      for (int i = 0; i < 32; ++i) m |= (v[i] >= theta ? 1u : 0u) << i;
      const int valid = args.Ncols - col0;
      if (valid < 32) m &= (1u << valid) - 1u;
      if (!row_ok) m = 0u;
      mask[c] = m;
      total += __popc(m);
    }
  }
  if (!__any_sync(0xffffffffu, total > 0)) return;
  int pos = 0;
  if (total > 0) pos = atomicAdd(&args.cand_cnt[row], total);
  const int64_t base = static_cast<int64_t>(row) * args.cand_cap;
#pragma unroll
  for (int c = 0; c < kBNMax / 32; ++c) {
    if (!__any_sync(0xffffffffu, mask[c] != 0u)) continue;  // warp-uniform
    float v[32];
    __syncwarp();
    tmem_ld32(tacc + 32 * c, v);
    // one iteration per passing logit of the lane that has the most in this chunk
    uint32_t m = mask[c];
    while (__any_sync(0xffffffffu, m != 0u)) {
      const bool has = m != 0u;
      const int i = has ? __ffs(m) - 1 : 0;
      const float val = select32(v, i);
      if (has) {
        if (pos < args.cand_cap) {
          args.cand_val[base + pos] = val;
          args.cand_id[base + pos] = col_tile + 32 * c + i;
        }
        ++pos;
        m &= m - 1u;
      }
    }
  }
}

template <int EPI, bool A_MN, bool B_MN, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    kd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  using G = Geo<PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // A fallback launch that is not needed returns at once (the flag is the same for
  // both CTAs of a pair, so neither waits for the other).
  if (args.run_if != nullptr && *args.run_if == 0) return;
  // The forward's and the candidates' epilogues send nothing through shared memory,
  // so on a CTA pair the staging area becomes one more ring stage (same total).
  constexpr bool kStaging = (EPI != kEpiFwd && EPI != kEpiCand) || !PAIR;
  constexpr int kStages = kStaging ? G::kStages : G::kStages + kFwdExtraStages;
  static_assert(kStaging || kFwdExtraStages * G::kStageBytes <= kStagingBytes, "ring fits");
  uint8_t* staging = smem + kStages * G::kStageBytes;  // 1024-byte aligned
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + (kStaging ? kStagingBytes : 0));
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* acc_full = empty_bar + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Sched& sc = args.sched;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 = the pair's MMA issuer
  const int64_t unit0 = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t unit_step = PAIR ? (gridDim.x >> 1) : gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], PAIR ? 8 : 4);  // one arrive per epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (uses_tma_out<EPI>(args)) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(tmem_slot, kTmemCols);
    tmem_relinquish<PAIR>();
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // the peer's copies and arrives target barriers initialised above
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Give up in this CTA and, for a pair, in the peer too.
  auto raise_abort = [&]() {
    *abort_flag = 1;
    if constexpr (PAIR)
      st_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u), 1u);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t u = unit0; ok && u < sc.total; u += unit_step) {
        const Unit d = sched_unit(sc, u);
        const int m_rows = d.m_blk * G::kTileRows + static_cast<int>(rank) * kBM;  // this CTA's A rows
        for (int nb = d.n_begin; ok && nb < d.n_end; ++nb) {
          const int n_cols = nb * args.BN + (PAIR ? static_cast<int>(rank) * (args.BN / 2) : 0);
          for (int kb = d.kb_begin; kb < d.kb_end; ++kb) {
            if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, args.timeout_ns,
                                   args.status, 6)) {
              ok = false;
              raise_abort();
              break;
            }
            uint8_t* a_dst = smem + stage * G::kStageBytes;
            uint8_t* b_dst = a_dst + G::kAStageBytes;
            const int k0 = kb * kBK;
            if constexpr (PAIR) {
              // both CTAs' copies complete on the first CTA's full barrier
              const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0u);
              if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * G::kStageBytes);
              if (!A_MN) {
                tma_load_2d_pair(a_dst, &tmA, fb, k0, m_rows + args.a_row_off);
              } else {
                tma_load_2d_pair(a_dst, &tmA, fb, m_rows, k0);
                tma_load_2d_pair(a_dst + kSlabBytes, &tmA, fb, m_rows + 64, k0);
              }
              if (!B_MN) {
                tma_load_2d_pair(b_dst, &tmB, fb, k0, n_cols);
              } else {
                tma_load_2d_pair(b_dst, &tmB, fb, n_cols, k0 + args.b_k_off);
                tma_load_2d_pair(b_dst + kSlabBytes, &tmB, fb, n_cols + 64, k0 + args.b_k_off);
              }
            } else {
              mbar_arrive_expect_tx(&full_bar[stage], G::kStageBytes);
              if (!A_MN) {
                tma_load_2d(a_dst, &tmA, &full_bar[stage], k0, m_rows + args.a_row_off);
              } else {
                tma_load_2d(a_dst, &tmA, &full_bar[stage], m_rows, k0);
                tma_load_2d(a_dst + kSlabBytes, &tmA, &full_bar[stage], m_rows + 64, k0);
              }
              if (!B_MN) {
                tma_load_2d(b_dst, &tmB, &full_bar[stage], k0, n_cols);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  tma_load_2d(b_dst + j * kSlabBytes, &tmB, &full_bar[stage], n_cols + 64 * j,
                              k0 + args.b_k_off);
              }
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (first CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool any_mma = false;
      const uint32_t a_lbo = A_MN ? kSlabBytes : 16;
      const uint32_t b_lbo = B_MN ? kSlabBytes : 16;
      const uint32_t a_kstep = A_MN ? 16 * 128 : 32;  // bytes per 16-deep k step
      const uint32_t b_kstep = B_MN ? 16 * 128 : 32;
      for (int64_t u = unit0; ok && u < sc.total; u += unit_step) {
        const Unit d = sched_unit(sc, u);
        for (int nb = d.n_begin; ok && nb < d.n_end; ++nb) {
          if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag, args.timeout_ns,
                                 args.status, 6)) {
            ok = false;
            raise_abort();
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBNMax);
          for (int kb = d.kb_begin; kb < d.kb_end; ++kb) {
            if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, args.timeout_ns,
                                   args.status, 6)) {
              ok = false;
              raise_abort();
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + stage * G::kStageBytes);
            const uint32_t b_addr = a_addr + G::kAStageBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint64_t adesc = umma_smem_desc(a_addr + k * a_kstep, a_lbo, 1024);
              const uint64_t bdesc = umma_smem_desc(b_addr + k * b_kstep, b_lbo, 1024);
              umma_bf16<PAIR>(d_tmem, adesc, bdesc, args.idesc,
                              (kb > d.kb_begin || k > 0) ? 1u : 0u);
            }
            any_mma = true;
            umma_commit<PAIR>(&empty_bar[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit<PAIR>(&acc_full[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      if (!ok && any_mma) {
        // Let every issued MMA finish before TMEM is released.
        umma_commit<PAIR>(drain_bar);
        volatile int no_abort = 0;
        mbar_wait_bounded(drain_bar, 0, &no_abort, 100000000ull, args.status, 6);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM sub-partition this warp may read
    const int row_in_tile = static_cast<int>(rank) * kBM + q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t acc_empty_addr0 =
        PAIR ? mapa_shared(smem_u32(&acc_empty[0]), 0u) : smem_u32(&acc_empty[0]);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const int K = args.K;
    const bool tma_out = uses_tma_out<EPI>(args);
    uint8_t* my_staging = staging + q * 2 * kOutChunkBytes;
    int sent = 0;  // chunks sent through TMA by this warp (selects the staging buffer)
    for (int64_t u = unit0; ok && u < sc.total; u += unit_step) {
      const Unit d = sched_unit(sc, u);
      const int m0 = d.m_blk * G::kTileRows;
      const int row = m0 + row_in_tile;          // local output row
      const bool row_ok = row < args.M;
      // per-unit state
      float m2 = -INFINITY, s2 = 0.0f;           // fwd running (max, sum) in base 2
      int ptr = 0;
      int2 cur = make_int2(INT_MAX, 0);          // current entry of the sorted teacher list
      int64_t rowK = 0;
      float gs = 0.0f, lse2 = 0.0f;
      bool dz_row = false;
      if (EPI == kEpiFwd && row_ok) {
        rowK = (args.row_base + row) * K;
        ptr = lower_bound_id(args.pairs + rowK, K, d.n_begin * args.BN);
        cur.x = (ptr < K) ? __ldg(&args.pairs[rowK + ptr].x) : INT_MAX;
      }
      if (EPI == kEpiDz && row_ok) {
        const int64_t g = args.row_base + row;
        dz_row = (args.mask == nullptr) || (args.mask[g] != 0);
        if (dz_row) {
          gs = __ldg(&args.dloss[g]) * args.inv_T;
          lse2 = __ldg(&args.lse[g]) * 1.4426950408889634f;
          rowK = g * K;
          ptr = lower_bound_id(args.pairs + rowK, K, d.n_begin * args.BN);
          cur = (ptr < K) ? __ldg(&args.pairs[rowK + ptr]) : make_int2(INT_MAX, 0);
        }
      }
      float theta = INFINITY;  // kEpiCand: nothing passes on a row past the end
      if (EPI == kEpiCand && row_ok) theta = __ldg(&args.thr[static_cast<int64_t>(row) * args.thr_stride +
                                                             args.thr_stride - 1]);
      if (EPI == kEpiDw && args.accumulate != 0 && row_ok) {
        // The L2 add at the end of this unit reads the tile's current dW values:
        // start bringing this row's part in from DRAM while the main loop runs.
        const int c0 = d.n_begin * args.BN;
        const int ncols = min(args.BN, args.Ncols - c0);
        const float* src = args.out_f32 + static_cast<int64_t>(row) * args.ld_out + c0;
        for (int c = 0; c < ncols; c += 32) prefetch_l2(src + c);
      }
      for (int nb = d.n_begin; nb < d.n_end; ++nb) {
        const bool got = mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag, args.timeout_ns,
                                           args.status, 6);
        if (!__all_sync(0xffffffffu, got)) {  // keep the warp's decision uniform
          ok = false;
          if (lane == 0) raise_abort();
          break;
        }
        tc_fence_after();
        const uint32_t tacc = lane_addr + static_cast<uint32_t>(acc * kBNMax);
        const int col_tile = nb * args.BN;
        if constexpr (EPI == kEpiCand) cand_tile(tacc, col_tile, theta, row, row_ok, args);
#pragma unroll 1
        for (int c = 0; c < (EPI == kEpiCand ? 0 : kBNMax / 32); ++c) {
          if (32 * c >= args.BN) break;
          const int col0 = col_tile + 32 * c;
          if (col0 >= args.Ncols) break;
          float v[32];
          __syncwarp();
          tmem_ld32(tacc + 32 * c, v);
          if constexpr (EPI == kEpiFwd) {
            while (cur.x < col0 + 32) {
              args.zk[rowK + ptr] = select32(v, cur.x - col0);
              ++ptr;
              cur.x = (ptr < K) ? __ldg(&args.pairs[rowK + ptr].x) : INT_MAX;
            }
            if (col0 + 32 > args.Ncols) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i >= args.Ncols) v[i] = -INFINITY;
            }
            float mx = v[0];
#pragma unroll
            for (int i = 1; i < 32; ++i) mx = fmaxf(mx, v[i]);
            const float mnew = fmaxf(m2, mx * args.scale2);
            // arguments and partial sums two lanes at a time (packed fp32x2); the four
            // partial sums take the same elements in the same order as scalar code would
            const uint64_t sc2 = f32x2(args.scale2, args.scale2), nm2 = f32x2(-mnew, -mnew);
            uint64_t p01 = f32x2(0.f, 0.f), p23 = f32x2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              p01 = add_f32x2(p01, ex2_f32x2(fma_f32x2(f32x2(v[i + 0], v[i + 1]), sc2, nm2)));
              p23 = add_f32x2(p23, ex2_f32x2(fma_f32x2(f32x2(v[i + 2], v[i + 3]), sc2, nm2)));
            }
            float a0, a1, a2, a3;
            f32x2_split(p01, a0, a1);
            f32x2_split(p23, a2, a3);
            s2 = s2 * ex2_approx(m2 - mnew) + ((a0 + a1) + (a2 + a3));
            m2 = mnew;
          } else if constexpr (EPI == kEpiDz) {
            float dv[32];
            if (dz_row) {
#pragma unroll
              for (int i = 0; i < 32; i += 2)
                f32x2_split(mul_f32x2(f32x2(gs, gs), ex2_f32x2(fma_f32x2(f32x2(v[i], v[i + 1]),
                                                                         f32x2(args.scale2, args.scale2),
                                                                         f32x2(-lse2, -lse2)))),
                            dv[i], dv[i + 1]);
              while (cur.x < col0 + 32) {
                sub_at32(dv, cur.x - col0, gs * __int_as_float(cur.y));
                ++ptr;
                cur = (ptr < K) ? __ldg(&args.pairs[rowK + ptr]) : make_int2(INT_MAX, 0);
              }
              if (col0 + 32 > args.Ncols) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col0 + i >= args.Ncols) dv[i] = 0.0f;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) dv[i] = 0.0f;
            }
            // Rows past the chunk's end are stored as zeros (the dW contraction
            // reads them up to the next multiple of 64); columns past V are
            // clipped by the TMA unit and never read back.
            const int r0 = m0 + static_cast<int>(rank) * kBM + q * 32;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            send_chunk_bf16(&tmC, my_staging + (sent & 1) * kOutChunkBytes, dv, lane, col0, r0);
            ++sent;
          } else if (tma_out) {
            // dW, plain C, dH k-split partials: staged boxes, TMA store / add.
            // Boxes that start past the last row or column are not sent; the TMA
            // unit clips the rest at the tensor's edges.
            const int r0 = m0 + static_cast<int>(rank) * kBM + q * 32;  // warp-uniform
            const int rem = args.BN - 32 * c;  // columns of this tile left (multiple of 16)
            const int boxes = (rem >= 32 && col0 + kOutBoxCols < args.Ncols) ? 2 : 1;
            if (r0 < args.M) {
              const int y0 = (EPI == kEpiDh) ? r0 + d.slot * args.out_slot_rows : r0;
              if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous boxes are read
              __syncwarp();
              send_chunk(&tmC, my_staging + (sent & 1) * kOutChunkBytes, v, lane, col0, y0, boxes,
                         EPI == kEpiDw && args.accumulate != 0);
              ++sent;
            }
          } else if constexpr (EPI == kEpiDh) {
            if (row_ok) {
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                const int cg = col0 + 8 * g;
                if (32 * c + 8 * g < args.BN && cg < args.Ncols) {
                  uint4 w;
                  w.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
                  w.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
                  w.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
                  w.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
                  *reinterpret_cast<uint4*>(args.out_bf16 + (args.row_base + row) * args.Ncols + cg) = w;
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(acc_empty_addr0 + 8u * static_cast<uint32_t>(acc));
          else
            mbar_arrive(&acc_empty[acc]);
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (EPI == kEpiFwd && ok && row_ok)
        args.part[(args.row_base + row) * args.slots + d.slot] = make_float2(m2, s2);
    }
    // The output boxes must be fully written before the kernel ends (and before
    // the staging memory is released).
    if (tma_out && lane == 0) bulk_wait_group_all();
  }

  if (*abort_flag) {
    // Bulk copies and MMAs already issued by this CTA or its peer complete within
    // microseconds; give them a millisecond before shared memory and TMEM go away.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<PAIR>(tmem_base, kTmemCols);
}

}  // namespace kd
