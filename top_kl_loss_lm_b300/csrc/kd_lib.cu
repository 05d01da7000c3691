// kd_lib.cu — host side of libkdtopk: argument checks, workspace plan, TMA
// descriptors, and the launch sequence of the forward and backward.
//
// Forward  (one pass over the vocabulary, nothing tokens x vocabulary stored):
//   prep -> per 4,096 rows: fused GEMM + online logsumexp + top-K gather -> combine
// Backward (the logits are recomputed, C tokens at a time):
//   prep -> for each group of kDwGroup chunks:
//             for each chunk: GEMM + dZ epilogue (the chunk's dZ slot, bf16)
//                             -> dH = dZ W  (split over V, fixed-order sum)
//             dW (+)= dZ^T H over the group's tokens
// Also: the loss from materialised logits (kd_topk_kl_logits) and the teacher's
// top-K cache (kd_teacher_topk: logit GEMM per chunk + exact per-row selection).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>  // header-only: ranges reach a profiler when one is attached

#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "../../include/kd_topk_kl.h"
#include "../../include/kd_topk_kl_testing.h"
#include "kd_aux.cuh"
#include "kd_gemm.cuh"
#include "kd_logits.cuh"
#include "kd_topk_cache.cuh"
#include "kd_sched.h"

namespace kd {

namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
  bool ready = false;
  bool ok = false;
  unsigned long long ctx_id = 0;  // the CUDA context the values below belong to
  int dev = 0;
  int num_sms = 0;
  int pair_slots = 0;     // CTA pairs of the GEMM kernel that fit on the device at once
  int* status = nullptr;  // device address of g_kd_status
};

// Every GEMM of the loss runs on CTA pairs (cta_group::2, 256-row tiles).
constexpr bool kPair = true;
constexpr int kTileRows = Geo<kPair>::kTileRows;

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Driver entry points used to tell CUDA contexts apart: a device's cached
// addresses (the status word, the allocation-free forward's scratch) belong to
// the context that was current when they were looked up, and are looked up
// again when that context has gone (cudaDeviceReset) and another has replaced it.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

void* driver_entry(const char* name, unsigned version) {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return fn;
  cudaGetLastError();
  return nullptr;
}

// Unique id of the calling thread's current context; 0 when there is none yet
// (the runtime creates the device's primary context on its first real use).
unsigned long long current_ctx_id() {
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr ||
      g_ctx_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Every kernel launch of the library sits in an NVTX range named for its
// category (seen by Nsight tools; a no-op without one). Optional per-launch
// timing (test hook kd_debug_profile): a start/stop event pair recorded on the
// launching stream around every kernel of the library.
enum ProfCat : int { kProfPrep = 0, kProfFwdGemm, kProfCombine, kProfDzGemm, kProfDhGemm, kProfDhSum,
                     kProfDwGemm, kProfLogits, kProfTopkGemm, kProfTopkSelect, kProfTranspose,
                     kProfCats };
struct Prof {
  bool on = false;
  std::vector<cudaEvent_t> ev;      // pool: 2 per record
  std::vector<int> cat;             // category of record i
  size_t used = 0;
};
Prof g_prof;

const char* const kProfNames[kProfCats] = {"kd prep", "kd fwd gemm", "kd combine", "kd dZ gemm",
                                           "kd dH gemm", "kd dH sum", "kd dW gemm", "kd logits",
                                           "kd topk gemm", "kd topk select", "kd transpose"};

struct ProfScope {
  cudaStream_t s;
  int rec = -1;
  ProfScope(int c, cudaStream_t st) : s(st) {
    nvtxRangePushA(kProfNames[c]);
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_prof.used * 2 + 2 > g_prof.ev.size()) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
        cudaGetLastError();
        return;
      }
      g_prof.ev.push_back(a);
      g_prof.ev.push_back(b);
    }
    rec = static_cast<int>(g_prof.used++);
    if (g_prof.cat.size() < g_prof.used) g_prof.cat.resize(g_prof.used);
    g_prof.cat[rec] = c;
    cudaEventRecord(g_prof.ev[2 * rec], s);
  }
  ~ProfScope() {
    if (rec >= 0) cudaEventRecord(g_prof.ev[2 * rec + 1], s);
    nvtxRangePop();
  }
};

const DevInfo* device_info(kd_status* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *err = KD_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ctx_current) {
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent", 4000));
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId", 12000));
  }
  DevInfo& d = g_dev[dev];
  unsigned long long cur = current_ctx_id();
  if (cur == 0 && d.ready) {
    // no current context, e.g. after cudaDeviceReset: have the runtime set up the
    // device's primary context now, so that it can be told apart from the old one
    if (cudaSetDevice(dev) == cudaSuccess) cur = current_ctx_id();
    cudaGetLastError();
  }
  if (!d.ready || cur != d.ctx_id) {
    d.ready = true;
    d.dev = dev;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    void* p = nullptr;
    const bool sym = cudaGetSymbolAddress(&p, g_kd_status) == cudaSuccess;
    d.status = static_cast<int*>(p);
    if (!g_encode)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(
          driver_entry("cuTensorMapEncodeTiled", 12000));
    d.ok = sym && g_encode != nullptr && major == 10 && minor == 3 && d.num_sms > 0;
    d.pair_slots = d.num_sms / 2;
    if (d.ok) {
      auto kern = kd_gemm_kernel<kEpiPlain, false, false, true>;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes) ==
          cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(d.num_sms & ~1));
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = kGemmSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0 &&
            n < d.pair_slots)
          d.pair_slots = n;
      }
    }
    cudaGetLastError();
    d.ctx_id = current_ctx_id();  // the symbol lookup above made the context current
  }
  if (!d.ok) {
    *err = KD_ERR_UNSUPPORTED;
    return nullptr;
  }
  return &d;
}

// 2D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// `row_bytes` between rows, box of box_inner x box_outer, 128-byte swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  std::memset(m, 0, sizeof(*m));
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D output map for the TMA store / add epilogue: `cols` contiguous elements
// per row, `rows` rows, boxes of 32 rows x 64 bytes (16 fp32 or 32 bf16) with
// 64-byte swizzle.
bool make_out_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                  bool bf16 = false) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(bf16 ? 32 : kOutBoxCols), 32};
  cuuint32_t es[2] = {1, 1};
  std::memset(m, 0, sizeof(*m));
  return g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Layout {
  // shared by forward and backward
  size_t pairs = 0, ent = 0;
  // forward
  size_t part = 0, zk = 0;
  // backward
  size_t dz = 0, ht = 0, dhp = 0;
  int64_t ldht = 0;  // row stride (elements) of the transposed H copy
  size_t fwd_end = 0, bwd_end = 0, total = 0;
  int slots = 0;
  int64_t C = 0, C_pad = 0, dz_ld = 0;
  int NB = 0;
  int G = 1;  // backward chunks per dW launch (dZ slots kept at once)
};

// Backward chunks whose dZ is kept together so that one dW launch contracts over
// all their tokens: half as many read-add-write passes over the fp32 dW.
constexpr int kDwGroup = 2;
constexpr int kMaxDwGroup = 4;


Layout plan(int64_t N, int D, int V, int K, int64_t chunk) {
  Layout L;
  L.NB = static_cast<int>(cdiv(V, kBNMax));
  L.slots = L.NB < kMaxSlots ? L.NB : kMaxSlots;
  size_t off = 0;
  L.pairs = off;
  off = align256(off + static_cast<size_t>(N) * K * sizeof(int2));
  L.ent = off;
  off = align256(off + static_cast<size_t>(N) * sizeof(float));
  const size_t common = off;
  // forward
  L.part = off;
  off = align256(off + static_cast<size_t>(N) * L.slots * sizeof(float2));
  L.zk = off;
  off = align256(off + static_cast<size_t>(N) * K * sizeof(float));
  L.fwd_end = off;
  // backward (reuses the forward's region)
  off = common;
  int64_t C = chunk <= 0 ? 4096 : chunk;
  C = cdiv(C, kTileRows) * kTileRows;
  const int64_t Nr = cdiv(N, kTileRows) * kTileRows;
  if (C > Nr) C = Nr;
  if (C < kTileRows) C = kTileRows;
  L.C = C;
  L.C_pad = C;
  L.dz_ld = static_cast<int64_t>(L.NB) * kBNMax;
  L.G = static_cast<int>(cdiv(N, C) < kDwGroup ? (cdiv(N, C) < 1 ? 1 : cdiv(N, C)) : kDwGroup);
  L.dz = off;
  off = align256(off + static_cast<size_t>(L.G) * L.C_pad * L.dz_ld * sizeof(uint16_t));
  // the dW group's H^T [D x G*C]: the K-major B operand of dW
  L.ldht = static_cast<int64_t>(L.G) * L.C_pad;
  L.ht = off;
  off = align256(off + static_cast<size_t>(D) * L.ldht * sizeof(uint16_t));
  L.dhp = off;  // k-split partials of dH take whatever follows (sized at call time)
  L.bwd_end = off;
  L.total = L.fwd_end > L.bwd_end ? L.fwd_end : L.bwd_end;
  return L;
}

// dH partial slices that fit in ws_bytes after the fixed backward layout.
int ksplit_that_fits(const Layout& L, int D, size_t ws_bytes, int wanted) {
  if (wanted <= 1) return 1;
  const size_t slice = static_cast<size_t>(L.C_pad) * D * sizeof(float);
  if (ws_bytes <= L.dhp) return 1;
  const size_t room = ws_bytes - L.dhp;
  int fit = static_cast<int>(room / slice);
  if (fit < 2) return 1;
  return fit < wanted ? fit : wanted;
}

int wanted_ksplit(int64_t C_pad, int D, int V, int grid) {
  const int MB = static_cast<int>(C_pad / kTileRows);
  const int bn = mn_major_tile_width(D);  // dH's hidden tiles (B = W, MN-major)
  const int NBd = static_cast<int>(cdiv(D, bn));
  const int KB = static_cast<int>(cdiv(V, kBK));
  return choose_ksplit(static_cast<int64_t>(MB) * NBd, KB, grid);
}

kd_status cuda_check() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

// dst [C x R] = transpose of src [R x C] (bf16; C a multiple of 8).
kd_status launch_transpose(const uint16_t* src, int64_t R, int C, int64_t lds, uint16_t* dst,
                           int64_t ldd, cudaStream_t s) {
  if (R <= 0) return KD_OK;
  ProfScope ps(kProfTranspose, s);
  const dim3 grid(static_cast<unsigned>(cdiv(R, kTrTile)), static_cast<unsigned>(cdiv(C, kTrTile)));
  kd_transpose_kernel<<<grid, 256, 0, s>>>(src, R, C, lds, dst, ldd);
  return cuda_check();
}

template <int EPI, bool AMN, bool BMN, bool PAIR>
kd_status launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                      const GemmArgs& args, const DevInfo* di, cudaStream_t s) {
  auto kern = kd_gemm_kernel<EPI, AMN, BMN, PAIR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_CUDA;
  }
  const int64_t slots = PAIR ? di->pair_slots : di->num_sms;
  const int64_t units = args.sched.total < slots ? args.sched.total : slots;
  if (units < 1) return KD_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * units : units));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a, b, c, args) != cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_CUDA;
  }
  return cuda_check();
}

// Rows per forward launch: kPanelRows row blocks (one schedule panel).
inline int64_t fwd_chunk_rows(int64_t N) {
  const int64_t fc = static_cast<int64_t>(kPanelRows) * kTileRows;
  return N < fc ? (N < 1 ? 1 : N) : fc;
}

// Persistent workers the GEMM schedules are planned for (CTA pairs).
inline int gemm_slots(const DevInfo* di) { return kPair ? di->pair_slots : di->num_sms; }

GemmArgs base_args(const DevInfo* di) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = di->status;
  a.timeout_ns = 2000000000ull;  // 2 s: far above any stage wait of a healthy pipeline
  return a;
}

// Whether every non-NULL pointer in the list addresses memory the current device
// can use: device memory of that device, or managed memory.
bool on_device(const DevInfo* di, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (p == nullptr) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (a.type == cudaMemoryTypeManaged) continue;
    if (a.type != cudaMemoryTypeDevice || a.device != di->dev) return false;
  }
  return true;
}

kd_status check_common(const uint16_t* H, const uint16_t* W, const int32_t* idx, const float* t,
                       int64_t N, int D, int V, int K, float T, const void* ws) {
  if (N < 0 || D <= 0 || V <= 0 || K < 1 || K > kMaxTopK) return KD_ERR_ARG;
  if (D % 8 != 0) return KD_ERR_ARG;
  if (!(T > 0.0f) || !std::isfinite(T)) return KD_ERR_ARG;
  if (N > (int64_t(1) << 31) - kBM || V > (1 << 30)) return KD_ERR_UNSUPPORTED;
  if (N == 0) return KD_OK;
  if (!H || !W || !idx || !t || !ws) return KD_ERR_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(ws, 256) || !aligned(idx, 4) || !aligned(t, 4))
    return KD_ERR_ALIGN;
  return KD_OK;
}

}  // namespace
}  // namespace kd

using namespace kd;

namespace kd {
namespace {

// The vocabulary columns a call covers: ids [v0, v0 + Vs) of a vocabulary of V
// (the whole vocabulary is v0 = 0, Vs = V; a vocabulary shard of W otherwise).
struct VRange {
  int v0, Vs, V;
};

// Workspace bytes for the forward and backward over Vs vocabulary columns. An
// fp32 dH (a vocabulary shard's partial) needs at least one slice of partials.
size_t workspace_bytes(int64_t N, int D, int Vs, int K, int64_t chunk, bool dh_f32) {
  Layout L = plan(N, D, Vs, K, chunk);
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) sms = n;
  }
  cudaGetLastError();
  const int ks = wanted_ksplit(L.C_pad, D, Vs, kPair ? sms / 2 : sms);
  size_t bwd = L.bwd_end;
  if (ks > 1 || dh_f32) bwd = align256(L.dhp + static_cast<size_t>(ks) * L.C_pad * D * sizeof(float));
  return L.fwd_end > bwd ? L.fwd_end : bwd;
}

// Forward over the columns of vr. Whole vocabulary: loss and lse per row. A
// shard (shard_out set): per row (lse over the shard, sum_k P_k z_k over the
// shard's teacher entries) into shard_out and the teacher grid's entropy into
// ent_out; loss and lse are not written.
kd_status fwd_run(const DevInfo* di, const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                  const float* topk_logit, const uint8_t* mask, int64_t N, int D, VRange vr, int K,
                  float T, float* loss, float* lse, int64_t* n_valid, float2* shard_out,
                  float* ent_out, void* ws, size_t ws_bytes, cudaStream_t s) {
  kd_status st = KD_OK;
  if (cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s) != cudaSuccess) return KD_ERR_CUDA;
  if (N == 0) return KD_OK;
  const int V = vr.Vs;  // the GEMM's vocabulary columns
  const Layout L = plan(N, D, V, K, 0);
  if (ws_bytes < L.fwd_end) return KD_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int2* pairs = reinterpret_cast<int2*>(w + L.pairs);
  float* ent = ent_out ? ent_out : reinterpret_cast<float*>(w + L.ent);
  float2* part = reinterpret_cast<float2*>(w + L.part);
  float* zk = reinterpret_cast<float*>(w + L.zk);
  const float inv_T = 1.0f / T;

  {
    ProfScope ps(kProfPrep, s);
    kd_prep_kernel<<<static_cast<unsigned>(cdiv(N, kPrepWarps)), kPrepWarps * 32, 0, s>>>(
        topk_idx, topk_logit, mask, N, K, vr.V, vr.v0, vr.Vs, inv_T, pairs, ent,
        reinterpret_cast<unsigned long long*>(n_valid), di->status);
  }
  if ((st = cuda_check()) != KD_OK) return st;

  CUtensorMap mH, mW;
  if (!make_map(&mH, H, D, N, static_cast<uint64_t>(D) * 2, kBK, kBM) ||
      !make_map(&mW, W, D, V, static_cast<uint64_t>(D) * 2, kBK, Geo<kPair>::kBRows))
    return KD_ERR_CUDA;
  const int KB = static_cast<int>(cdiv(D, kBK));
  GemmArgs a = base_args(di);
  a.Ncols = V;
  a.BN = kBNMax;
  a.idesc = umma_idesc_bf16(kTileRows, kBNMax, false, false);
  a.K = K;
  a.scale2 = 1.4426950408889634f * inv_T;
  a.inv_T = inv_T;
  a.pairs = pairs;
  a.zk = zk;
  a.part = part;
  a.slots = L.slots;
  // One launch per row chunk: the 74 CTA pairs then share the chunk's H rows
  // and each W tile in L2, instead of spreading over rows from several panels.
  const int64_t FC = fwd_chunk_rows(N);
  int S_full = 0, S_last = 0;
  const int64_t last_start = ((N - 1) / FC) * FC;
  for (int64_t c0 = 0; c0 < N; c0 += FC) {
    const int64_t rows = (N - c0) < FC ? (N - c0) : FC;
    a.sched = make_panel_sched(static_cast<int>(cdiv(rows, kTileRows)), L.NB, KB, gemm_slots(di));
    a.M = static_cast<int>(rows);
    a.a_row_off = static_cast<int>(c0);
    a.row_base = c0;
    if (a.sched.P != 1) return KD_ERR_UNSUPPORTED;  // one panel per chunk by construction
    if (c0 == 0) S_full = a.sched.S0;
    if (c0 == last_start) S_last = a.sched.S0;
    ProfScope ps(kProfFwdGemm, s);
    if ((st = launch_gemm<kEpiFwd, false, false, kPair>(mH, mW, mH, a, di, s)) != KD_OK) return st;
  }
  {
    ProfScope ps(kProfCombine, s);
    kd_combine_kernel<<<static_cast<unsigned>(cdiv(N, 256)), 256, 0, s>>>(
        last_start, S_full, S_last, part, L.slots, pairs, zk, ent, mask, N, K, V, inv_T, loss, lse,
        shard_out);
  }
  return cuda_check();
}

// Backward over the columns of vr. dH is written as bf16 (dH) or, for a
// vocabulary shard's partial, as fp32 (dH_f32, added to its contents if
// accumulate_dH); dW covers the vr.Vs columns.
kd_status bwd_run(const DevInfo* di, const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                  const float* topk_logit, const uint8_t* mask, const float* lse,
                  const float* dloss, int64_t N, int D, VRange vr, int K, float T,
                  int64_t chunk_tokens, int accumulate_dW, uint16_t* dH, float* dH_f32,
                  int accumulate_dH, float* dW, void* ws, size_t ws_bytes, cudaStream_t s) {
  kd_status st = KD_OK;
  const int V = vr.Vs;  // the GEMMs' vocabulary columns
  if (N == 0) {
    if (!accumulate_dW &&
        cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * D * sizeof(float), s) != cudaSuccess)
      return KD_ERR_CUDA;
    return KD_OK;
  }
  const bool f32 = dH_f32 != nullptr;
  const Layout L = plan(N, D, V, K, chunk_tokens);
  if (ws_bytes < L.bwd_end) return KD_ERR_WORKSPACE;
  const size_t slice = static_cast<size_t>(L.C_pad) * D * sizeof(float);
  if (f32 && ws_bytes < L.dhp + slice) return KD_ERR_WORKSPACE;
  const int KS = ksplit_that_fits(L, D, ws_bytes, wanted_ksplit(L.C_pad, D, V, gemm_slots(di)));
  const bool partials = KS > 1 || f32;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int2* pairs = reinterpret_cast<int2*>(w + L.pairs);
  float* ent = reinterpret_cast<float*>(w + L.ent);
  uint16_t* dz = reinterpret_cast<uint16_t*>(w + L.dz);
  float* dhp = reinterpret_cast<float*>(w + L.dhp);
  const float inv_T = 1.0f / T;

  {
    ProfScope ps(kProfPrep, s);
    kd_prep_kernel<<<static_cast<unsigned>(cdiv(N, kPrepWarps)), kPrepWarps * 32, 0, s>>>(
        topk_idx, topk_logit, mask, N, K, vr.V, vr.v0, vr.Vs, inv_T, pairs, ent, nullptr,
        di->status);
  }
  if ((st = cuda_check()) != KD_OK) return st;

  // dH: B = W, MN-major, 256-wide hidden tiles (zero fill past D). dW: B = the
  // group's H^T, K-major, even hidden tiles (no padded columns). The transposed
  // copy of the 8,192-token group costs ~0.03 ms and made dW ~8% faster than
  // reading H MN-major with 256-wide padded tiles; a transposed W for dH gained
  // less than its transpose cost.
  const int BNh = mn_major_tile_width(D);
  const int NBh = static_cast<int>(cdiv(D, BNh));
  const int BNw = hidden_tile_width(D);
  const int NBw = static_cast<int>(cdiv(D, BNw));
  if (L.G < 1 || L.G > kMaxDwGroup) return KD_ERR_UNSUPPORTED;
  uint16_t* ht = reinterpret_cast<uint16_t*>(w + L.ht);

  CUtensorMap mH_k, mW_k, mW_mn, mDz_mn;
  CUtensorMap mDz_k[kMaxDwGroup], mDz_out[kMaxDwGroup];  // one per dZ slot
  const uint64_t rowH = static_cast<uint64_t>(D) * 2;
  const uint64_t rowDz = static_cast<uint64_t>(L.dz_ld) * 2;
  const int64_t slot_elems = L.C_pad * L.dz_ld;
  if (!make_map(&mH_k, H, D, N, rowH, kBK, kBM) ||
      !make_map(&mW_k, W, D, V, rowH, kBK, Geo<kPair>::kBRows) ||
      !make_map(&mW_mn, W, D, V, rowH, 64, kBK) ||
      !make_map(&mDz_mn, dz, V, static_cast<uint64_t>(L.G) * L.C_pad, rowDz, 64, kBK))
    return KD_ERR_CUDA;
  for (int g = 0; g < L.G; ++g)
    if (!make_map(&mDz_k[g], dz + g * slot_elems, V, L.C_pad, rowDz, kBK, kBM) ||
        !make_out_map(&mDz_out[g], dz + g * slot_elems, V, L.C_pad, rowDz, true))
      return KD_ERR_CUDA;
  CUtensorMap mDw_out, mDhp_out;
  if (!make_out_map(&mDw_out, dW, D, V, static_cast<uint64_t>(D) * 4) ||
      (partials && !make_out_map(&mDhp_out, dhp, D, static_cast<uint64_t>(KS) * L.C_pad,
                                 static_cast<uint64_t>(D) * 4)))
    return KD_ERR_CUDA;
  if (!partials) mDhp_out = mDw_out;  // unused: dH is written in bf16 directly

  const int KBd = static_cast<int>(cdiv(D, kBK));
  const int KBv = static_cast<int>(cdiv(V, kBK));
  const int MBv = static_cast<int>(cdiv(V, kTileRows));
  const int64_t group = static_cast<int64_t>(L.G) * L.C;
  for (int64_t g0 = 0; g0 < N; g0 += group) {
   const int64_t group_rows = (N - g0) < group ? (N - g0) : group;
   for (int slot = 0; slot < L.G && g0 + slot * L.C < N; ++slot) {
    const int64_t c0 = g0 + slot * L.C;
    const int64_t rows = (N - c0) < L.C ? (N - c0) : L.C;
    const int MBc = static_cast<int>(cdiv(rows, kTileRows));

    // 1. recompute the chunk's logits, dZ epilogue -> dz (bf16)
    GemmArgs a = base_args(di);
    a.sched = make_panel_sched(MBc, L.NB, KBd, gemm_slots(di));
    a.M = static_cast<int>(rows);
    a.Ncols = V;
    a.BN = kBNMax;
    a.idesc = umma_idesc_bf16(kTileRows, kBNMax, false, false);
    a.a_row_off = static_cast<int>(c0);
    a.row_base = c0;
    a.K = K;
    a.scale2 = 1.4426950408889634f * inv_T;
    a.inv_T = inv_T;
    a.pairs = pairs;
    a.lse = lse;
    a.dloss = dloss;
    a.mask = mask;
    a.dz = dz;
    a.dz_ld = L.dz_ld;
    {
      ProfScope ps(kProfDzGemm, s);
      if ((st = launch_gemm<kEpiDz, false, false, kPair>(mH_k, mW_k, mDz_out[slot], a, di, s)) !=
          KD_OK)
        return st;
    }

    // 2. dH rows of the chunk = dZ W (contraction over V, split KS ways)
    GemmArgs h = base_args(di);
    h.sched = make_tile_sched(MBc, NBh, KBv, KS);
    h.M = static_cast<int>(rows);
    h.Ncols = D;
    h.BN = BNh;
    h.idesc = umma_idesc_bf16(kTileRows, BNh, false, true);
    h.row_base = c0;
    h.out_bf16 = dH;
    h.out_f32 = dhp;
    h.part_stride = L.C_pad * static_cast<int64_t>(D);
    h.out_slot_rows = static_cast<int>(L.C_pad);
    h.dh_partials = f32 ? 1 : 0;
    {
      ProfScope ps(kProfDhGemm, s);
      if ((st = launch_gemm<kEpiDh, false, true, kPair>(mDz_k[slot], mW_mn, mDhp_out, h, di, s)) !=
          KD_OK)
        return st;
    }
    if (partials) {
      const int64_t groups = rows * (D / 8);
      int64_t blocks = cdiv(groups, 256);
      if (blocks > 8L * di->num_sms) blocks = 8L * di->num_sms;
      ProfScope ps(kProfDhSum, s);
      if (f32)
        kd_dh_sum_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            dhp, h.sched.KS, h.part_stride, rows, D, dH_f32 + c0 * D, accumulate_dH);
      else
        kd_dh_sum_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            dhp, h.sched.KS, h.part_stride, rows, D, dH + c0 * D, 0);
      if ((st = cuda_check()) != KD_OK) return st;
    }

   }
    // 3. dW (+)= dZ^T H over the group's tokens: slot g's rows are tokens
    //    g0 + g*C + t, so the stacked slots are the group's tokens in order (rows
    //    past the end of a short last chunk were stored as zeros). B is the
    //    group's H^T [D x tokens]; its map ends at the group's last token, so the
    //    k-blocks past it read zeros.
    if ((st = launch_transpose(H + g0 * D, group_rows, D, D, ht, L.ldht, s)) != KD_OK) return st;
    CUtensorMap mHt_k;
    if (!make_map(&mHt_k, ht, group_rows, D, static_cast<uint64_t>(L.ldht) * 2, kBK,
                  Geo<kPair>::kBRows))
      return KD_ERR_CUDA;
    GemmArgs g = base_args(di);
    g.sched = make_tile_sched(MBv, NBw, static_cast<int>(cdiv(group_rows, kBK)), 1);
    g.M = V;
    g.Ncols = D;
    g.BN = BNw;
    g.idesc = umma_idesc_bf16(kTileRows, BNw, true, false);
    g.out_f32 = dW;
    g.ld_out = D;
    g.accumulate = (g0 > 0 || accumulate_dW) ? 1 : 0;
    {
      ProfScope ps(kProfDwGemm, s);
      if ((st = launch_gemm<kEpiDw, true, false, kPair>(mDz_mn, mHt_k, mDw_out, g, di, s)) != KD_OK)
        return st;
    }
  }
  return KD_OK;
}

// Checks shared by the vocabulary-shard calls: the range lies in [0, V).
bool shard_range_ok(int v0, int V_shard, int V) {
  return v0 >= 0 && V_shard >= 1 && V_shard <= V && v0 <= V - V_shard;
}

}  // namespace
}  // namespace kd

extern "C" size_t kd_topk_kl_workspace_size(int64_t N, int D, int V, int K, int64_t chunk_tokens) {
  if (N < 0 || D <= 0 || V <= 0 || K < 1 || K > kMaxTopK || D % 8 != 0) return 0;
  return workspace_bytes(N, D, V, K, chunk_tokens, false);
}

extern "C" kd_status kd_topk_kl_fwd(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                                    const float* topk_logit, const uint8_t* mask, int64_t N, int D,
                                    int V, int K, float T, float* loss, float* lse,
                                    int64_t* n_valid, void* ws, size_t ws_bytes,
                                    kd_stream_t stream) {
  kd_status st = check_common(H, W, topk_idx, topk_logit, N, D, V, K, T, ws);
  if (st != KD_OK) return st;
  if (!n_valid || (N > 0 && (!loss || !lse))) return KD_ERR_ARG;
  if (!aligned(n_valid, 8) || !aligned(loss, 4) || !aligned(lse, 4)) return KD_ERR_ALIGN;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {n_valid}) ||
      (N > 0 && !on_device(di, {H, W, topk_idx, topk_logit, mask, loss, lse, ws})))
    return KD_ERR_ARG;
  return fwd_run(di, H, W, topk_idx, topk_logit, mask, N, D, VRange{0, V, V}, K, T, loss, lse,
                 n_valid, nullptr, nullptr, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kd_status kd_topk_kl_bwd(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                                    const float* topk_logit, const uint8_t* mask, const float* lse,
                                    const float* dloss, int64_t N, int D, int V, int K, float T,
                                    int64_t chunk_tokens, int accumulate_dW, uint16_t* dH,
                                    float* dW, void* ws, size_t ws_bytes, kd_stream_t stream) {
  kd_status st = check_common(H, W, topk_idx, topk_logit, N, D, V, K, T, ws);
  if (st != KD_OK) return st;
  if (!dW || (N > 0 && (!lse || !dloss || !dH))) return KD_ERR_ARG;
  if (!aligned(dW, 16) || !aligned(dH, 16) || !aligned(lse, 4) || !aligned(dloss, 4))
    return KD_ERR_ALIGN;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {dW}) ||
      (N > 0 && !on_device(di, {H, W, topk_idx, topk_logit, mask, lse, dloss, dH, ws})))
    return KD_ERR_ARG;
  return bwd_run(di, H, W, topk_idx, topk_logit, mask, lse, dloss, N, D, VRange{0, V, V}, K, T,
                 chunk_tokens, accumulate_dW, dH, nullptr, 0, dW, ws, ws_bytes,
                 reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ vocabulary shards

extern "C" size_t kd_topk_kl_shard_workspace_size(int64_t N, int D, int V_shard, int K,
                                                  int64_t chunk_tokens) {
  if (N < 0 || D <= 0 || V_shard <= 0 || K < 1 || K > kMaxTopK || D % 8 != 0) return 0;
  return workspace_bytes(N, D, V_shard, K, chunk_tokens, true);
}

extern "C" kd_status kd_topk_kl_fwd_shard(const uint16_t* H, const uint16_t* W_shard, int v0,
                                          int V_shard, int V, const int32_t* topk_idx,
                                          const float* topk_logit, const uint8_t* mask, int64_t N,
                                          int D, int K, float T, float* parts, float* ent,
                                          int64_t* n_valid, void* ws, size_t ws_bytes,
                                          kd_stream_t stream) {
  kd_status st = check_common(H, W_shard, topk_idx, topk_logit, N, D, V, K, T, ws);
  if (st != KD_OK) return st;
  if (!shard_range_ok(v0, V_shard, V)) return KD_ERR_ARG;
  if (!n_valid || (N > 0 && (!parts || !ent))) return KD_ERR_ARG;
  if (!aligned(n_valid, 8) || !aligned(parts, 8) || !aligned(ent, 4)) return KD_ERR_ALIGN;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {n_valid}) ||
      (N > 0 && !on_device(di, {H, W_shard, topk_idx, topk_logit, mask, parts, ent, ws})))
    return KD_ERR_ARG;
  return fwd_run(di, H, W_shard, topk_idx, topk_logit, mask, N, D, VRange{v0, V_shard, V}, K, T,
                 nullptr, nullptr, n_valid, reinterpret_cast<float2*>(parts), ent, ws, ws_bytes,
                 reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kd_status kd_topk_kl_shard_merge(const float* parts, int R, const float* ent,
                                            const uint8_t* mask, int64_t N, float T, float* loss,
                                            float* lse, kd_stream_t stream) {
  if (N < 0 || R < 1 || !(T > 0.0f) || !std::isfinite(T)) return KD_ERR_ARG;
  if (N == 0) return KD_OK;
  if (!parts || !ent || !loss || !lse) return KD_ERR_ARG;
  if (!aligned(parts, 8) || !aligned(ent, 4) || !aligned(loss, 4) || !aligned(lse, 4))
    return KD_ERR_ALIGN;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {parts, ent, mask, loss, lse})) return KD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ProfScope ps(kProfCombine, s);
  kd_shard_merge_kernel<<<static_cast<unsigned>(cdiv(N, 256)), 256, 0, s>>>(
      reinterpret_cast<const float2*>(parts), R, ent, mask, N, 1.0f / T, loss, lse);
  return cuda_check();
}

extern "C" kd_status kd_topk_kl_bwd_shard(const uint16_t* H, const uint16_t* W_shard, int v0,
                                          int V_shard, int V, const int32_t* topk_idx,
                                          const float* topk_logit, const uint8_t* mask,
                                          const float* lse, const float* dloss, int64_t N, int D,
                                          int K, float T, int64_t chunk_tokens, int accumulate_dW,
                                          int accumulate_dH, float* dH, float* dW_shard, void* ws,
                                          size_t ws_bytes, kd_stream_t stream) {
  kd_status st = check_common(H, W_shard, topk_idx, topk_logit, N, D, V, K, T, ws);
  if (st != KD_OK) return st;
  if (!shard_range_ok(v0, V_shard, V)) return KD_ERR_ARG;
  if (!dW_shard || (N > 0 && (!lse || !dloss || !dH))) return KD_ERR_ARG;
  if (!aligned(dW_shard, 16) || !aligned(dH, 16) || !aligned(lse, 4) || !aligned(dloss, 4))
    return KD_ERR_ALIGN;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {dW_shard}) ||
      (N > 0 && !on_device(di, {H, W_shard, topk_idx, topk_logit, mask, lse, dloss, dH, ws})))
    return KD_ERR_ARG;
  return bwd_run(di, H, W_shard, topk_idx, topk_logit, mask, lse, dloss, N, D,
                 VRange{v0, V_shard, V}, K, T, chunk_tokens, accumulate_dW, nullptr, dH,
                 accumulate_dH, dW_shard, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ mean-loss gradient

extern "C" kd_status kd_topk_kl_mean_grad(const float* loss, const uint8_t* mask, int64_t N,
                                          const int64_t* n_valid, float* dloss, double* loss_sum,
                                          kd_stream_t stream) {
  if (N < 0 || !n_valid || (!dloss && !loss_sum) || (loss_sum && N > 0 && !loss))
    return KD_ERR_ARG;
  if (!aligned(n_valid, 8) || !aligned(loss, 4) || !aligned(dloss, 4) || !aligned(loss_sum, 8))
    return KD_ERR_ALIGN;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {loss, mask, n_valid, dloss, loss_sum})) return KD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ProfScope ps(kProfCombine, s);
  kd_mean_grad_kernel<<<1, kMeanThreads, 0, s>>>(loss_sum ? loss : nullptr, mask, N, n_valid, dloss,
                                                  loss_sum);
  return cuda_check();
}

// ------------------------------------------------------------------ loss from materialised logits

namespace kd {
namespace {

// Columns per CTA slice for a cluster of `cl` CTAs: a multiple of 64 so each slice
// starts on a 128-byte line.
inline int logits_slice(int V, int cl) { return static_cast<int>(cdiv(cdiv(V, cl), 64) * 64); }

constexpr size_t kLogitsSmemLimit = 227 * 1024;
static_assert(kMaxTopK <= kLogitsMaxK, "the logits kernel stages every teacher entry of a row");

// Shape of the loss-from-logits kernel. With the gradient: the smallest cluster
// whose slices, two row buffers each, let two CTAs of 256 compute threads share
// an SM (two independent row pipelines per SM keep enough bytes in flight: 78%
// of the HBM copy bandwidth at V = 201,088 against 67% with one CTA per SM and
// 49% with a four-buffer ring), else the smallest that fits one CTA per SM.
// Loss only: one row buffer and 128 compute threads per CTA, four CTAs per SM
// (80% against 65% with the gradient's shape). Returns false if nothing fits.
struct LogitsShape {
  int cl, nbuf, threads;
};
bool logits_shape(int V, bool grad, LogitsShape* out) {
  const int nbuf = grad ? 2 : 1;
  const int threads = grad ? kLogitsThreads : kLogitsThreadsLossOnly;
  for (int per_sm = grad ? 2 : 4; per_sm >= 1; per_sm = per_sm > 2 ? 2 : per_sm - 1)
    for (int cl = 1; cl <= kLogitsMaxCluster; cl *= 2)
      if (per_sm * logits_smem_bytes(logits_slice(V, cl), nbuf) <= kLogitsSmemLimit) {
        *out = {cl, nbuf, threads};
        return true;
      }
  return false;
}

template <int CL, int NBUF, int NT>
kd_status launch_logits(const LogitsArgs& a, const DevInfo* di, cudaStream_t s) {
  auto kern = kd_logits_kernel<CL, NBUF, NT>;
  const size_t smem = logits_smem_bytes(a.Vs, NBUF);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(di->num_sms / CL * CL));
  cfg.blockDim = dim3(NT + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
    cudaGetLastError();
    clusters = di->num_sms / CL;
  }
  int64_t want = a.N < clusters ? a.N : clusters;
  if (want < 1) return KD_OK;
  cfg.gridDim = dim3(static_cast<unsigned>(want * CL));
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_CUDA;
  }
  return cuda_check();
}

}  // namespace
}  // namespace kd

extern "C" size_t kd_topk_kl_logits_workspace_size(int64_t N, int K) {
  if (N < 0 || K < 1 || K > kMaxTopK) return 0;
  const size_t pairs = align256(static_cast<size_t>(N) * K * sizeof(int2));
  const size_t ent = align256(static_cast<size_t>(N) * sizeof(float));
  const size_t total = pairs + ent;
  return total > 0 ? total : 256;
}

extern "C" kd_status kd_topk_kl_logits(const uint16_t* Z, int64_t ldz, const int32_t* topk_idx,
                                       const float* topk_logit, const uint8_t* mask,
                                       const float* dloss, int64_t N, int V, int K, float T,
                                       float* loss, float* lse, int64_t* n_valid, uint16_t* dZ,
                                       int64_t lddz, void* ws, size_t ws_bytes,
                                       kd_stream_t stream) {
  if (N < 0 || V <= 0 || K < 1 || K > kMaxTopK || !(T > 0.0f) || !std::isfinite(T))
    return KD_ERR_ARG;
  if (N > (int64_t(1) << 40) || V > (1 << 30)) return KD_ERR_UNSUPPORTED;
  if (!n_valid) return KD_ERR_ARG;
  if (N > 0 && (!Z || !topk_idx || !topk_logit || !loss || !lse || !ws)) return KD_ERR_ARG;
  if (dZ && !dloss) return KD_ERR_ARG;
  if (ldz < V || (dZ && lddz < V)) return KD_ERR_ARG;
  if (V % 8 != 0 || ldz % 8 != 0 || (dZ && lddz % 8 != 0)) return KD_ERR_ALIGN;
  if (!aligned(Z, 16) || (dZ && !aligned(dZ, 16)) || !aligned(ws, 256) || !aligned(topk_idx, 4) ||
      !aligned(topk_logit, 4) || !aligned(loss, 4) || !aligned(lse, 4) || !aligned(n_valid, 8) ||
      (dloss && !aligned(dloss, 4)))
    return KD_ERR_ALIGN;
  LogitsShape shape;
  if (!logits_shape(V, dZ != nullptr, &shape)) return KD_ERR_UNSUPPORTED;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {n_valid}) ||
      (N > 0 && !on_device(di, {Z, topk_idx, topk_logit, mask, dloss, loss, lse, dZ, ws})))
    return KD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(n_valid, 0, sizeof(int64_t), s) != cudaSuccess) return KD_ERR_CUDA;
  if (N == 0) return KD_OK;
  if (ws_bytes < kd_topk_kl_logits_workspace_size(N, K)) return KD_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int2* pairs = reinterpret_cast<int2*>(w);
  float* ent = reinterpret_cast<float*>(w + align256(static_cast<size_t>(N) * K * sizeof(int2)));
  const float inv_T = 1.0f / T;
  {
    ProfScope ps(kProfPrep, s);
    kd_prep_kernel<<<static_cast<unsigned>(cdiv(N, kPrepWarps)), kPrepWarps * 32, 0, s>>>(
        topk_idx, topk_logit, mask, N, K, V, 0, V, inv_T, pairs, ent,
        reinterpret_cast<unsigned long long*>(n_valid), di->status);
  }
  if ((st = cuda_check()) != KD_OK) return st;
  LogitsArgs a;
  std::memset(&a, 0, sizeof(a));
  a.Z = Z;
  a.ldz = ldz;
  a.dZ = dZ;
  a.lddz = lddz;
  a.pairs = pairs;
  a.ent = ent;
  a.mask = mask;
  a.dloss = dloss;
  a.loss = loss;
  a.lse = lse;
  a.N = N;
  a.V = V;
  a.K = K;
  a.Vs = logits_slice(V, shape.cl);
  a.scale2 = 1.4426950408889634f * inv_T;
  a.inv_T = inv_T;
  a.status = di->status;
  a.timeout_ns = 2000000000ull;
  ProfScope ps(kProfLogits, s);
  if (shape.nbuf == 2 && shape.threads == kLogitsThreads) {  // with the gradient
    switch (shape.cl) {
      case 1: return launch_logits<1, 2, kLogitsThreads>(a, di, s);
      case 2: return launch_logits<2, 2, kLogitsThreads>(a, di, s);
      case 4: return launch_logits<4, 2, kLogitsThreads>(a, di, s);
      default: return launch_logits<8, 2, kLogitsThreads>(a, di, s);
    }
  }
  switch (shape.cl) {  // loss only
    case 1: return launch_logits<1, 1, kLogitsThreadsLossOnly>(a, di, s);
    case 2: return launch_logits<2, 1, kLogitsThreadsLossOnly>(a, di, s);
    case 4: return launch_logits<4, 1, kLogitsThreadsLossOnly>(a, di, s);
    default: return launch_logits<8, 1, kLogitsThreadsLossOnly>(a, di, s);
  }
}

// ------------------------------------------------------------------ teacher top-K cache

namespace kd {
namespace {
// Rows of teacher logits materialised at a time (fp32, one chunk of the workspace).
int64_t topk_chunk_rows(int64_t N) {
  const int64_t c = 16 * static_cast<int64_t>(kTileRows);  // 4,096
  return N < c ? cdiv(N < 1 ? 1 : N, kTileRows) * kTileRows : c;
}
inline int64_t topk_ld(int V) { return cdiv(V, 8) * 8; }

// Resident select CTAs per SM, with the carveout set to favour shared memory (the
// kernel's 35 KB of shared arrays would otherwise limit an SM to three CTAs).
int select_blocks_per_sm() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(kd_topk_select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kd_topk_select_kernel, kSelectThreads, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    cudaGetLastError();
  });
  return n;
}
}  // namespace
}  // namespace kd

namespace kd {
namespace {
// Vocabularies from this size on take the fused path: a threshold per row from a
// strided sample of W's rows, then the full GEMM keeps only the logits at or
// above it. Smaller ones materialise each chunk's logits and select from them.
constexpr int kFusedTopkMinV = 16384;

struct TopkPlan {
  int64_t C = 0, ldz = 0;      // rows per chunk, row stride of the materialised logits
  bool fused = false;
  int64_t stride = 1, S = 0, lds = 0;  // sample: W rows 0, stride, 2*stride, ... (S of them)
  int r = 0;                   // row threshold = the r-th largest sampled logit
  size_t zc = 0, zs = 0, wsm = 0, thr = 0, cv = 0, ci = 0, cnt = 0, flag = 0, total = 0;
};

TopkPlan topk_plan(int64_t N, int D, int V, int K) {
  TopkPlan P;
  P.C = topk_chunk_rows(N);
  P.ldz = topk_ld(V);
  size_t off = 0;
  P.zc = off;  // the materialised chunk: the small-vocabulary path and the fallback
  off = align256(off + static_cast<size_t>(P.C) * P.ldz * sizeof(float));
  P.fused = V >= kFusedTopkMinV;
  if (P.fused) {
    P.stride = V / 2048 < 32 ? (V / 2048 < 1 ? 1 : V / 2048) : 32;
    P.S = cdiv(V, P.stride);
    P.lds = topk_ld(static_cast<int>(P.S));
    // lambda = the expected number of the row's top K in the sample; the threshold
    // is the (lambda + 4 sqrt(lambda) + 8)-th largest sampled logit, so the kept set
    // misses a top-K logit (and the chunk falls back) about once in 1e10 rows for a
    // sample that behaves like a random one (12 at K = 100 left ~1e-4: one row in a
    // chunk of 4,096 then sent about every second chunk to the fallback)
    const int64_t lam = cdiv(static_cast<int64_t>(K) * P.S, V);
    const int64_t want = lam + static_cast<int64_t>(std::ceil(4.0 * std::sqrt(static_cast<double>(lam)))) + 8;
    P.r = static_cast<int>(want < P.S ? want : P.S);
    if (P.r > kThrMaxRank) {  // cannot happen for K <= 256 and a sampling stride >= 8
      P.fused = false;
      P.total = off;
      return P;
    }
    P.zs = off;
    off = align256(off + static_cast<size_t>(P.C) * P.lds * sizeof(float));
    P.wsm = off;
    off = align256(off + static_cast<size_t>(P.S) * D * sizeof(uint16_t));
    P.thr = off;
    off = align256(off + static_cast<size_t>(P.C) * sizeof(float));
    P.cv = off;
    off = align256(off + static_cast<size_t>(P.C) * kCandCap * sizeof(float));
    P.ci = off;
    off = align256(off + static_cast<size_t>(P.C) * kCandCap * sizeof(int32_t));
    P.cnt = off;
    off = align256(off + static_cast<size_t>(P.C) * sizeof(int));
    P.flag = off;
    off = align256(off + sizeof(int));
  }
  P.total = off;
  return P;
}

kd_status launch_select(const float* Z, int64_t ldz, int64_t rows, int V, int K, int32_t* idx,
                        float* val, const int* run_if, const DevInfo* di, cudaStream_t s) {
  // persistent: as many CTAs as are resident at once (each CTA loops over rows)
  int64_t grid = static_cast<int64_t>(select_blocks_per_sm()) * di->num_sms;
  if (grid > rows) grid = rows;
  ProfScope ps(kProfTopkSelect, s);
  kd_topk_select_kernel<<<static_cast<unsigned>(grid), kSelectThreads, 0, s>>>(Z, ldz, rows, V, K,
                                                                              idx, val, run_if);
  return cuda_check();
}
}  // namespace
}  // namespace kd

extern "C" size_t kd_teacher_topk_workspace_size(int64_t N, int D, int V, int K) {
  if (N < 0 || D <= 0 || D % 8 != 0 || V <= 0 || K < 1 || K > kSelectMaxK || K > V) return 0;
  return topk_plan(N, D, V, K).total;
}

extern "C" kd_status kd_teacher_topk(const uint16_t* H, const uint16_t* W, int64_t N, int D, int V,
                                     int K, int32_t* topk_idx, float* topk_logit, void* ws,
                                     size_t ws_bytes, kd_stream_t stream) {
  if (N < 0 || D <= 0 || V <= 0 || K < 1 || K > kSelectMaxK || K > V || D % 8 != 0)
    return KD_ERR_ARG;
  if (N > (int64_t(1) << 31) - kBM || V > (1 << 30)) return KD_ERR_UNSUPPORTED;
  if (N == 0) return KD_OK;
  if (!H || !W || !topk_idx || !topk_logit || !ws) return KD_ERR_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(ws, 256) || !aligned(topk_idx, 4) ||
      !aligned(topk_logit, 4))
    return KD_ERR_ALIGN;
  const TopkPlan P = topk_plan(N, D, V, K);
  if (ws_bytes < P.total) return KD_ERR_WORKSPACE;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {H, W, topk_idx, topk_logit, ws})) return KD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* Zc = reinterpret_cast<float*>(w + P.zc);
  CUtensorMap mH, mW, mZ;
  if (!make_map(&mH, H, D, N, static_cast<uint64_t>(D) * 2, kBK, kBM) ||
      !make_map(&mW, W, D, V, static_cast<uint64_t>(D) * 2, kBK, Geo<kPair>::kBRows) ||
      !make_out_map(&mZ, Zc, V, P.C, static_cast<uint64_t>(P.ldz) * 4))
    return KD_ERR_CUDA;
  const int NB = static_cast<int>(cdiv(V, kBNMax));
  const int KB = static_cast<int>(cdiv(D, kBK));

  float* Zs = reinterpret_cast<float*>(w + P.zs);
  uint16_t* Ws = reinterpret_cast<uint16_t*>(w + P.wsm);
  float* thr = reinterpret_cast<float*>(w + P.thr);
  float* cv = reinterpret_cast<float*>(w + P.cv);
  int32_t* ci = reinterpret_cast<int32_t*>(w + P.ci);
  int* cnt = reinterpret_cast<int*>(w + P.cnt);
  int* flag = reinterpret_cast<int*>(w + P.flag);
  CUtensorMap mWs, mZs;
  if (P.fused) {
    {
      ProfScope ps(kProfTranspose, s);  // the sample of W's rows, once per call
      const int64_t n = P.S * (D / 8);
      int64_t blocks = cdiv(n, 256);
      if (blocks > 8L * di->num_sms) blocks = 8L * di->num_sms;
      kd_gather_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(W, P.stride, P.S, D, Ws);
      if ((st = cuda_check()) != KD_OK) return st;
    }
    if (!make_map(&mWs, Ws, D, P.S, static_cast<uint64_t>(D) * 2, kBK, Geo<kPair>::kBRows) ||
        !make_out_map(&mZs, Zs, P.S, P.C, static_cast<uint64_t>(P.lds) * 4))
      return KD_ERR_CUDA;
  }

  for (int64_t c0 = 0; c0 < N; c0 += P.C) {
    const int64_t rows = (N - c0) < P.C ? (N - c0) : P.C;
    const int MB = static_cast<int>(cdiv(rows, kTileRows));
    int32_t* out_idx = topk_idx + c0 * K;
    float* out_val = topk_logit + c0 * K;
    GemmArgs a = base_args(di);
    a.sched = make_panel_sched(MB, NB, KB, gemm_slots(di));
    a.M = static_cast<int>(rows);
    a.Ncols = V;
    a.BN = kBNMax;
    a.idesc = umma_idesc_bf16(kTileRows, kBNMax, false, false);
    a.a_row_off = static_cast<int>(c0);
    if (P.fused) {
      // 1. the sampled logits and each row's threshold (its r-th largest sampled logit)
      GemmArgs sa = a;
      sa.sched = make_panel_sched(MB, static_cast<int>(cdiv(P.S, kBNMax)), KB, gemm_slots(di));
      sa.Ncols = static_cast<int>(P.S);
      {
        ProfScope ps(kProfTopkGemm, s);
        if ((st = launch_gemm<kEpiPlain, false, false, kPair>(mH, mWs, mZs, sa, di, s)) != KD_OK)
          return st;
      }
      {
        int64_t grid = cdiv(rows, kThrWarps);
        if (grid > 8L * di->num_sms) grid = 8L * di->num_sms;
        ProfScope ps(kProfTopkSelect, s);
        if (P.r <= 32)
          kd_row_threshold_kernel<true><<<static_cast<unsigned>(grid), kThrWarps * 32, 0, s>>>(
              Zs, P.lds, rows, static_cast<int>(P.S), P.r, thr);
        else
          kd_row_threshold_kernel<false><<<static_cast<unsigned>(grid), kThrWarps * 32, 0, s>>>(
              Zs, P.lds, rows, static_cast<int>(P.S), P.r, thr);
        if ((st = cuda_check()) != KD_OK) return st;
      }
      // 2. the full GEMM keeps what reaches the threshold
      if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(rows) * sizeof(int), s) != cudaSuccess ||
          cudaMemsetAsync(flag, 0, sizeof(int), s) != cudaSuccess)
        return KD_ERR_CUDA;
      GemmArgs ca = a;
      ca.thr = thr;
      ca.thr_stride = 1;
      ca.cand_val = cv;
      ca.cand_id = ci;
      ca.cand_cnt = cnt;
      ca.cand_cap = kCandCap;
      {
        ProfScope ps(kProfTopkGemm, s);
        if ((st = launch_gemm<kEpiCand, false, false, kPair>(mH, mW, mH, ca, di, s)) != KD_OK)
          return st;
      }
      // 3. the K largest of each row's candidates; a row whose list is short or
      //    overflowed raises the flag
      {
        int64_t grid = rows < 8L * di->num_sms ? rows : 8L * di->num_sms;
        ProfScope ps(kProfTopkSelect, s);
        kd_cand_select_kernel<<<static_cast<unsigned>(grid), kCandThreads, 0, s>>>(
            cv, ci, cnt, kCandCap, rows, K, out_idx, out_val, flag);
        if ((st = cuda_check()) != KD_OK) return st;
      }
      // 4. fallback for the chunk, run only if the flag is up: materialise and select
      a.run_if = flag;
    }
    {
      ProfScope ps(kProfTopkGemm, s);
      if ((st = launch_gemm<kEpiPlain, false, false, kPair>(mH, mW, mZ, a, di, s)) != KD_OK)
        return st;
    }
    if ((st = launch_select(Zc, P.ldz, rows, V, K, out_idx, out_val, P.fused ? flag : nullptr, di,
                            s)) != KD_OK)
      return st;
  }
  return KD_OK;
}

extern "C" kd_status kd_get_status(kd_stream_t stream) {
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KD_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KD_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KD_ERR_CUDA;
  return static_cast<kd_status>(v);
}

extern "C" const char* kd_status_string(kd_status status) {
  switch (status) {
    case KD_OK: return "ok";
    case KD_ERR_ARG: return "invalid argument (size, NULL pointer, temperature, or memory not on the current device)";
    case KD_ERR_ALIGN: return "pointer alignment violates the ABI rules";
    case KD_ERR_UNSUPPORTED: return "unsupported shape or device (needs an sm_103 GPU)";
    case KD_ERR_WORKSPACE: return "workspace smaller than kd_topk_kl_workspace_size()";
    case KD_ERR_INDEX: return "teacher id outside [0, V) at a counted row";
    case KD_ERR_TIMEOUT: return "bounded pipeline wait ran out; results are invalid";
    case KD_ERR_CUDA: return "CUDA runtime or driver call failed";
    case KD_ERR_BOUNDS: return "checked build: a device-side bounds check failed (access skipped)";
  }
  return "unknown status";
}

// ------------------------------------------------------------------ test hooks

extern "C" kd_status kd_debug_gemm_bf16(const uint16_t* A, const uint16_t* B, float* C, int M, int N,
                                        int K, int a_mn, int b_mn, int cta_pair, kd_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || M % 8 || N % 8 || K % 8) return KD_ERR_ARG;
  if (!A || !B || !C) return KD_ERR_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return KD_ERR_ALIGN;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (!on_device(di, {A, B, C})) return KD_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool pair = cta_pair != 0;
  const int rows = pair ? Geo<true>::kTileRows : Geo<false>::kTileRows;
  const int b_rows = pair ? Geo<true>::kBRows : Geo<false>::kBRows;
  // K-major B: the even split of the dH / dW products (e.g. 12 x 240 for N = 2,880);
  // MN-major B: see mn_major_tile_width
  const int BN = b_mn ? mn_major_tile_width(N) : hidden_tile_width(N);
  CUtensorMap ma, mb;
  bool ok;
  if (!a_mn)
    ok = make_map(&ma, A, K, M, static_cast<uint64_t>(K) * 2, kBK, kBM);
  else
    ok = make_map(&ma, A, M, K, static_cast<uint64_t>(M) * 2, 64, kBK);
  if (!b_mn)
    ok = ok && make_map(&mb, B, K, N, static_cast<uint64_t>(K) * 2, kBK, b_rows);
  else
    ok = ok && make_map(&mb, B, N, K, static_cast<uint64_t>(N) * 2, 64, kBK);
  CUtensorMap mc;
  ok = ok && make_out_map(&mc, C, N, M, static_cast<uint64_t>(N) * 4);
  if (!ok) return KD_ERR_CUDA;
  GemmArgs a = base_args(di);
  a.sched = make_tile_sched(static_cast<int>(cdiv(M, rows)), static_cast<int>(cdiv(N, BN)),
                            static_cast<int>(cdiv(K, kBK)), 1);
  a.M = M;
  a.Ncols = N;
  a.BN = BN;
  a.idesc = umma_idesc_bf16(rows, BN, a_mn != 0, b_mn != 0);
  a.out_f32 = C;
  a.ld_out = N;
  if (pair) {
    if (!a_mn && !b_mn) return launch_gemm<kEpiPlain, false, false, true>(ma, mb, mc, a, di, s);
    if (!a_mn && b_mn) return launch_gemm<kEpiPlain, false, true, true>(ma, mb, mc, a, di, s);
    if (a_mn && !b_mn) return launch_gemm<kEpiPlain, true, false, true>(ma, mb, mc, a, di, s);
    return launch_gemm<kEpiPlain, true, true, true>(ma, mb, mc, a, di, s);
  }
  if (!a_mn && !b_mn) return launch_gemm<kEpiPlain, false, false, false>(ma, mb, mc, a, di, s);
  if (!a_mn && b_mn) return launch_gemm<kEpiPlain, false, true, false>(ma, mb, mc, a, di, s);
  if (a_mn && !b_mn) return launch_gemm<kEpiPlain, true, false, false>(ma, mb, mc, a, di, s);
  return launch_gemm<kEpiPlain, true, true, false>(ma, mb, mc, a, di, s);
}

extern "C" kd_status kd_debug_wait_timeout(uint64_t timeout_ns, kd_stream_t stream) {
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  if (timeout_ns > 2000000000ull) timeout_ns = 2000000000ull;
  kd_wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(timeout_ns, di->status);
  return cuda_check();
}

extern "C" kd_status kd_debug_schedule(int kind, int64_t rows, int64_t cols, int64_t depth,
                                       int grid_units, int tile_rows, int32_t* counts, int64_t* info) {
  if (rows <= 0 || cols <= 0 || depth <= 0 || grid_units <= 0 || kind < 0 || kind > 2 || !info ||
      (tile_rows != 128 && tile_rows != 256))
    return KD_ERR_ARG;
  const int num_sms = grid_units;
  const int MB = static_cast<int>(cdiv(rows, tile_rows));
  const int KB = static_cast<int>(cdiv(depth, kBK));
  int BN, NB;
  Sched sc;
  if (kind == 0) {
    BN = kBNMax;
    NB = static_cast<int>(cdiv(cols, BN));
    sc = make_panel_sched(MB, NB, KB, num_sms);
  } else {
    // dH reads W MN-major (256-wide hidden tiles), dW the group's H^T K-major (even tiles)
    BN = kind == 1 ? mn_major_tile_width(static_cast<int>(cols)) : hidden_tile_width(static_cast<int>(cols));
    NB = static_cast<int>(cdiv(cols, BN));
    const int ks = (kind == 1) ? choose_ksplit(static_cast<int64_t>(MB) * NB, KB, num_sms) : 1;
    sc = make_tile_sched(MB, NB, KB, ks);
  }
  const int64_t grid = sc.total < num_sms ? sc.total : num_sms;
  int max_slot = 0;
  for (int64_t u = 0; u < sc.total; ++u) {
    const Unit d = sched_unit(sc, u);
    if (d.slot + 1 > max_slot) max_slot = d.slot + 1;
    if (counts)
      for (int nb = d.n_begin; nb < d.n_end; ++nb)
        for (int kb = d.kb_begin; kb < d.kb_end; ++kb)
          counts[(static_cast<int64_t>(d.m_blk) * NB + nb) * KB + kb] += 1;
  }
  info[0] = sc.total;
  info[1] = grid;
  info[2] = MB;
  info[3] = NB;
  info[4] = KB;
  info[5] = BN;
  info[6] = max_slot;
  info[7] = sc.KS;
  return KD_OK;
}

extern "C" kd_status kd_debug_profile(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof.on = enable != 0;
  g_prof.used = 0;
  return KD_OK;
}

extern "C" kd_status kd_debug_profile_read(double* total_ms, int64_t* launches, int n) {
  if (!total_ms || !launches || n < 1) return KD_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < n; ++i) {
    total_ms[i] = 0.0;
    launches[i] = 0;
  }
  for (size_t r = 0; r < g_prof.used; ++r) {
    if (cudaEventSynchronize(g_prof.ev[2 * r + 1]) != cudaSuccess) {
      cudaGetLastError();
      return KD_ERR_CUDA;
    }
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * r], g_prof.ev[2 * r + 1]) != cudaSuccess) {
      cudaGetLastError();
      return KD_ERR_CUDA;
    }
    const int c = g_prof.cat[r];
    if (c < n) {
      total_ms[c] += ms;
      launches[c] += 1;
    }
  }
  g_prof.used = 0;
  return KD_OK;
}

// ------------------------------------------------------------------ forward without allocation
//
// For callers that cannot allocate device memory themselves: a plugin that
// runs inside a host process whose allocator has already reserved the GPU's
// memory, or a latency-critical path where cudaMalloc (which may synchronise
// the device) is not allowed. The forward's scratch lives in this fixed array
// instead of a caller workspace. The array is part of the library's device
// image, so every GPU that loads the library holds its 64 MiB until the
// process exits.
namespace {
constexpr size_t kFwdScratchBytes = size_t(64) << 20;
}  // namespace

static __device__ __align__(256) unsigned char g_kd_fwd_scratch[kFwdScratchBytes];

namespace {
std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx = 0;  // context the address was looked up in
  void* ptr = nullptr;
};
ScratchAddr g_scratch[kd::kMaxDevices];
}  // namespace

extern "C" kd_status kd_topk_kl_fwd_noalloc(const uint16_t* H, const uint16_t* W,
                                            const int32_t* topk_idx, const float* topk_logit,
                                            const uint8_t* mask, int64_t N, int D, int V, int K,
                                            float T, float* loss, float* lse, int64_t* n_valid,
                                            kd_stream_t stream) {
  if (N < 0 || D <= 0 || V <= 0 || K < 1 || K > kMaxTopK || D % 8 != 0) return KD_ERR_ARG;
  if (plan(N, D, V, K, 0).fwd_end > kFwdScratchBytes) return KD_ERR_WORKSPACE;
  kd_status st = KD_OK;
  const DevInfo* di = device_info(&st);
  if (!di) return st;
  void* ws = nullptr;
  {
    // Set-up once per device (again if the device's context was replaced), with
    // that device current: the host-side name of the array is not a device
    // address, so ask the runtime for the real one.
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr& sa = g_scratch[di->dev];
    if (sa.ptr == nullptr || sa.ctx != di->ctx_id) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_kd_fwd_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return KD_ERR_CUDA;
      }
      sa.ptr = p;
      sa.ctx = di->ctx_id;
    }
    ws = sa.ptr;
  }
  return kd_topk_kl_fwd(H, W, topk_idx, topk_logit, mask, N, D, V, K, T, loss, lse, n_valid, ws,
                        kFwdScratchBytes, stream);
}
