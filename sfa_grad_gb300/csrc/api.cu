// C-ABI entry points (include/sfa_grad.h): validation, workspace plan and the
// launch sequence of the backward and the companion forward.
//
// aclnnSparseFlashAttentionGrad doc: 函数原型 (two-phase call), 参数说明
// (shapes, dtypes), 返回值 (status codes), 约束说明 (empty query, determinism),
// 规格约束 (supported ranges).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include <cudaTypedefs.h>

#include "sfa_grad.h"
#include "common.cuh"
#include "kernels.h"

namespace sfa {
namespace {

constexpr size_t kAlign = 256;
constexpr size_t kPdsCap = size_t(8) << 30;    // P + dS staging per token chunk
constexpr size_t kPartCap = size_t(8) << 30;   // deterministic partial rows (bf16) per chunk
constexpr int kAccRow = 1088;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  int layout, B, S1, S2, T1, T2, G, Gp, Kidx, bs, Keff, Kpad, mode, has_rope, det, is_f16;
  int Gs;    // heads per staged P / dS row (G rounded up to 16)
  int kvb;   // key-major dK / dV for block-sparse indices (kvb.cu)
  float scale;
  unsigned long long wait_ns;   // limit of every pipeline wait in the kernels
  int chunk;
  size_t off_err, off_batch, off_meta, off_dsum, off_acc, off_P, off_dS, off_rows, off_part, off_dscr, off_tstats;
  size_t off_bcnt, off_bcur, off_bgrp, off_bbeg, off_bng, off_bent, off_bres;
  size_t total;
};

sfa_status validate(const sfa_params* p, bool fwd, Plan* out) {
  if (!p) return SFA_ERR_NULLPTR;
  if (p->dtype != SFA_DTYPE_BF16 && p->dtype != SFA_DTYPE_FP16) return SFA_ERR_PARAM_INVALID;
  if (p->layout != SFA_LAYOUT_BSND && p->layout != SFA_LAYOUT_TND) return SFA_ERR_PARAM_INVALID;
  if (p->N2 != 1 || p->D != 512 || (p->Dr != 64 && p->Dr != 0)) return SFA_ERR_SHAPE;
  if (p->N1 < 1 || p->N1 > 128) return SFA_ERR_SHAPE;
  if (p->sparse_mode != 0 && p->sparse_mode != 3) return SFA_ERR_SHAPE;
  const int64_t bs = p->sparse_block_size;
  if (bs != 1 && bs != 8 && bs != 16 && bs != 32 && bs != 64) return SFA_ERR_SHAPE;
  if (p->K < 1 || p->K > (1 << 20)) return SFA_ERR_SHAPE;
  if (!std::isfinite(p->scale)) return SFA_ERR_SHAPE;
  if (p->deterministic != 0 && p->deterministic != 1) return SFA_ERR_PARAM_INVALID;
  if (p->wait_limit_us < 0) return SFA_ERR_PARAM_INVALID;
  if (p->B < 1) return SFA_ERR_SHAPE;
  int64_t T1, T2;
  if (p->layout == SFA_LAYOUT_BSND) {
    if (p->S1 < 0 || p->S2 < 0) return SFA_ERR_SHAPE;
    T1 = p->B * p->S1;
    T2 = p->B * p->S2;
  } else {
    if (p->T1 < 0 || p->T2 < 0) return SFA_ERR_SHAPE;
    T1 = p->T1;
    T2 = p->T2;
  }
  const int64_t keff = p->K * bs;
  if (keff > (1 << 24) || T1 > INT32_MAX / 2 || T2 > INT32_MAX / 2 || T1 * p->N1 > INT32_MAX / 2)
    return SFA_ERR_SHAPE;
  Plan& P = *out;
  std::memset(&P, 0, sizeof(P));
  P.layout = (int)p->layout;
  P.B = (int)p->B;
  P.S1 = (int)p->S1;
  P.S2 = (int)p->S2;
  P.T1 = (int)T1;
  P.T2 = (int)T2;
  P.G = (int)p->N1;
  P.Gp = P.G <= 64 ? 64 : 128;
  P.Gs = (P.G + 15) / 16 * 16;
  P.Kidx = (int)p->K;
  P.bs = (int)bs;
  P.Keff = (int)keff;
  P.Kpad = (int)((keff + 127) / 128 * 128);
  P.mode = (int)p->sparse_mode;
  P.has_rope = p->Dr == 64;
  P.det = fwd ? 0 : p->deterministic;
  P.is_f16 = p->dtype == SFA_DTYPE_FP16;
  P.scale = (float)p->scale;
  P.wait_ns = p->wait_limit_us > 0 ? (unsigned long long)p->wait_limit_us * 1000ull : kWaitNsDefault;
  // Block-sparse indices selected by many tokens: group the (token, index)
  // pairs by block start and accumulate each block's dK / dV in tensor memory
  // (one accumulator write per block instead of one reduction per pair).
  // Used when blocks hold >= 16 keys, at most 64 heads, and the average kv
  // row is selected by >= 8 query tokens.  Deterministic mode sorts each
  // group's pairs and adds the groups in bs launches (one per start residue
  // modulo bs, whose blocks share no key row).  The companion forward scores
  // the same groups per block (statistics, then P) and forms O per token with
  // the features on the MMA's rows.
  P.kvb = P.bs >= 16 && P.Gp == 64 && T2 > 0 && T1 * keff >= 8 * T2;
  // token chunking keeps the per-chunk staging bounded
  const size_t pds_per_tok = (size_t)P.Kpad * P.Gs * 2 * (fwd ? 1 : 2);
  size_t chunk = kPdsCap / pds_per_tok;
  if (P.det && !P.kvb) {
    const size_t part_per_tok = (size_t)P.Kpad * kAccRow * 2;
    const size_t c2 = kPartCap / part_per_tok;
    if (c2 < chunk) chunk = c2;
  }
  if (chunk < 1) chunk = 1;
  if (chunk > (size_t)P.T1) chunk = P.T1 > 0 ? P.T1 : 1;
  P.chunk = (int)chunk;
  size_t o = 0;
  P.off_err = o; o += up(16);
  P.off_batch = o; o += up((size_t)(2 * P.B + 2) * 4);
  P.off_meta = o; o += up((size_t)P.T1 * sizeof(TokMeta));
  P.off_dsum = o; o += fwd ? 0 : up((size_t)P.T1 * P.G * 4);
  P.off_acc = o; o += fwd ? 0 : up((size_t)P.T2 * kAccRow * 4);
  P.off_P = o; o += up(chunk * P.Kpad * P.Gs * 2);
  P.off_dS = o; o += fwd ? 0 : up(chunk * P.Kpad * P.Gs * 2);
  P.off_rows = o; o += P.kvb ? 0 : up(chunk * P.Kpad * 4);   // the key-major block plan reads no row table
  const size_t ents = chunk * (P.kvb ? P.Kidx : P.Kpad);   // sorted entries per chunk
  P.off_part = o; o += P.det && !P.kvb ? up(chunk * P.Kpad * kAccRow * 2) : 0;
  P.off_dscr = o; o += P.det ? up(2 * ents * 4) : 0;   // padded copies of long segments
  // forward partial statistics: per key tile of 128, or per block index
  P.off_tstats = o; o += fwd ? up(chunk * (P.kvb ? P.Kidx : P.Kpad / 32) * P.G * 2 * 4) : 0;
  // counting-sort bins: block starts + bs (key-major blocks) or kv rows
  // (deterministic reduction), and the sorted entries
  const bool bins = P.kvb || P.det;
  const size_t nb = bins ? (size_t)P.T2 + P.bs : 0;
  P.off_bcnt = o; o += bins ? up(nb * 4) : 0;
  P.off_bcur = o; o += bins ? up(nb * 4) : 0;
  P.off_bgrp = o; o += bins ? up(nb * 4) : 0;
  P.off_bbeg = o; o += bins ? up((nb + 1) * 4) : 0;
  P.off_bng = o; o += bins ? up(4) : 0;
  P.off_bent = o; o += bins ? up(ents * 4) : 0;
  P.off_bres = o; o += P.kvb ? up(64 * 4) : 0;
  P.total = o;
  return SFA_OK;
}

Prob make_prob(const Plan& P, uint8_t* ws) {
  Prob pr;
  std::memset(&pr, 0, sizeof(pr));
  pr.T1 = P.T1;
  pr.T2 = P.T2;
  pr.G = P.G;
  pr.Gp = P.Gp;
  pr.Gs = P.Gs;
  pr.Kidx = P.Kidx;
  pr.bs = P.bs;
  pr.Keff = P.Keff;
  pr.Kpad = P.Kpad;
  pr.has_rope = P.has_rope;
  pr.scale = P.scale;
  pr.wait_ns = P.wait_ns;
  pr.meta = reinterpret_cast<const TokMeta*>(ws + P.off_meta);
  pr.rowtab = reinterpret_cast<int*>(ws + P.off_rows);
  return pr;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on libcuda).
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

// 2-D row-major map over `rows` x `cols` 16-bit elements, box of box_cols
// columns x box_rows rows: 64 columns with 128-byte swizzle, or 32 columns
// with 64-byte swizzle.
bool encode2d(CUtensorMap* m, bool f16, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
              uint32_t box_cols = 64) {
  EncodeTiled fn = encoder();
  if (!fn) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (T1*G rows x 512) viewed as (64 features, rows, 8 panels): a box of `rows`
// head rows covers all eight 64-feature panels, panel after panel.
bool encode_panels3d(CUtensorMap* m, bool f16, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeTiled fn = encoder();
  if (!fn) return false;
  if (rows == 0) rows = 1;
  cuuint64_t dims[3] = {64, rows, 8};
  cuuint64_t strides[2] = {512 * 2, 64 * 2};
  cuuint32_t box[3] = {64, box_rows, 8};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Maps of the key-major block kernel: head rows with boxes of GK = G rounded
// up to 16 rows (one token's heads), staged P^T / dS^T as in Maps.
bool make_blk_maps(BlkMaps* M, const Plan& P, const void* q, const void* qr, const void* dO, const void* Pst,
                   const void* dSst) {
  const bool f = P.is_f16;
  const uint64_t TG = (uint64_t)P.T1 * P.G, R = (uint64_t)P.chunk * P.Kpad;
  const uint32_t gk = (uint32_t)((P.G + 15) / 16 * 16);
  bool ok = encode_panels3d(&M->q, f, q, TG, gk);
  ok = ok && encode2d(&M->qr, f, qr ? qr : q, qr ? 64 : 512, TG, gk);
  ok = ok && encode_panels3d(&M->dO, f, dO, TG, gk);
  ok = ok && encode2d(&M->P, f, Pst, P.Gs, R, 64);
  ok = ok && encode2d(&M->dS, f, dSst, P.Gs, R, 64);
  return ok;
}

// Maps of one call.  Tensors a call does not use (dO and dS in the forward,
// the rope pair without rope) alias a used tensor and are never read.
bool make_maps(Maps* M, const Plan& P, const void* q, const void* qr, const void* dO, const void* k, const void* kr,
               const void* v, const void* Pst, const void* dSst, const void* dq = nullptr,
               const void* dqr = nullptr, const void* part = nullptr) {
  const bool f = P.is_f16;
  const uint64_t TG = (uint64_t)P.T1 * P.G, T2 = (uint64_t)P.T2, R = (uint64_t)P.chunk * P.Kpad;
  bool ok = encode2d(&M->q, f, q, 512, TG, P.Gp);
  ok = ok && encode2d(&M->qr, f, qr ? qr : q, qr ? 64 : 512, TG, P.Gp);
  ok = ok && encode2d(&M->dO, f, dO ? dO : q, 512, TG, P.Gp);
  // key / value rows: one box = one selected block of bs rows (block-sparse
  // indices, bs >= 8); unused with single-key indices
  const uint32_t kb = P.bs >= 8 ? (uint32_t)P.bs : 1u;
  ok = ok && encode2d(&M->k, f, k, 512, T2, kb);
  ok = ok && encode2d(&M->kr, f, kr ? kr : k, kr ? 64 : 512, T2, kb);
  ok = ok && encode2d(&M->v, f, v, 512, T2, kb);
  ok = ok && encode2d(&M->P, f, Pst, P.Gs, R, 64);
  ok = ok && encode2d(&M->dS, f, dSst ? dSst : Pst, P.Gs, R, 64);
  ok = ok && encode2d(&M->Pw, f, Pst, P.Gs, R, 32, 32);
  ok = ok && encode2d(&M->dSw, f, dSst ? dSst : Pst, P.Gs, R, 32, 32);
  // the backward's dQ / dQRope outputs (the forward has none: aliases, unused)
  ok = ok && encode2d(&M->dQw, f, dq ? dq : q, 512, TG, 32, 32);
  ok = ok && encode2d(&M->dQRw, f, dqr ? dqr : (dq ? dq : q), dqr ? 64 : 512, TG, 32, 32);
  // deterministic partial rows (bf16 whatever the input type; the unused
  // map of the other plans aliases q)
  if (part) {
    EncodeTiled fn = encoder();
    cuuint64_t dims[2] = {(cuuint64_t)kAccRow, R == 0 ? 1 : R};
    cuuint64_t strides[1] = {(cuuint64_t)kAccRow * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    ok = ok && fn && fn(&M->partw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(part), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  } else {
    ok = ok && encode2d(&M->partw, f, q, 512, TG, 32, 32);
  }
  const uint32_t gk = (uint32_t)((P.G + 15) / 16 * 16);
  ok = ok && encode2d(&M->qg, f, q, 512, TG, gk);
  ok = ok && encode2d(&M->qrg, f, qr ? qr : q, qr ? 64 : 512, TG, gk);
  ok = ok && encode2d(&M->dOg, f, dO ? dO : q, 512, TG, gk);
  return ok;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// Text of the last failing CUDA call on this thread (sfa_last_error_message).
thread_local char g_last_error[256] = "";

sfa_status fail(cudaError_t e, int line) {
  snprintf(g_last_error, sizeof(g_last_error), "%s (CUDA error %d) at api.cu:%d", cudaGetErrorString(e), (int)e, line);
  (void)cudaGetLastError();
  return SFA_ERR_RUNTIME;
}

}  // namespace

void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

namespace {

#define SFA_CK(x)                                   \
  do {                                              \
    const cudaError_t sfa_e_ = (x);                 \
    if (sfa_e_ != cudaSuccess) return ::sfa::fail(sfa_e_, __LINE__); \
  } while (0)

__global__ void decode_kernel(Prob p, int* rows_out) {
  const long long n = (long long)p.T1 * p.Keff;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / p.Keff), s = (int)(i - (long long)t * p.Keff);
    rows_out[i] = slot_row(p, p.meta[t], t, s);
  }
}

// Records the caller's timing events between launches (sfa_grad_profile).
struct Marks {
  void** ev = nullptr;
  int n = 0, next = 0;
  cudaError_t mark(cudaStream_t st) {
    if (!ev || next >= n) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(ev[next++]), st);
  }
};

// Key tiles per key-side work item.  The fp32 accumulator rows one batch's
// tokens reduce into span its KV extent (S2, or the mean TND segment).  When
// that stays well inside the 129 MB L2, token-major order is best (one group
// of all tiles).  Otherwise groups of four tiles run tile-group major, so
// that with sorted index lists the concurrent reductions share a narrow band
// of key rows.
int kvq_tile_group(const Plan& P) {
  const int64_t rows = P.layout == SFA_LAYOUT_BSND ? (int64_t)P.S2 : (int64_t)P.T2 / (P.B > 0 ? P.B : 1);
  const int64_t bytes = rows * 1088 * 4;
  return bytes <= (int64_t)64 << 20 ? P.Kpad / 128 : 4;
}

// Kernel launches of one sfa_grad call, in order (sfa_grad_plan_names).
const char* const kChunkDet[] = {"rowtab", "sdp", "det_count", "det_scan", "det_scatter", "det_sort",
                                 "det_sort_long", "kvq", "det_reduce"};
const char* const kChunkKvq[] = {"rowtab", "sdp", "kvq"};
const char* const kChunkKvb[] = {"blk_count", "blk_scan", "blk_scatter", "sdpb", "kvb", "dqb"};
const char* const kChunkKvbDetHead[] = {"blk_count", "blk_scan", "blk_scatter", "blk_sort", "blk_sort_long", "sdpb"};

int64_t plan_names(const Plan& P, const char** out, int64_t cap) {
  int64_t n = 0;
  auto put = [&](const char* s) {
    if (n < cap && out) out[n] = s;
    ++n;
  };
  if (P.T1 == 0) return 0;
  if (P.layout == SFA_LAYOUT_TND) put("batch_prefix");
  put("meta");
  put("dsum");
  const int64_t chunks = (P.T1 + P.chunk - 1) / P.chunk;
  for (int64_t c = 0; c < chunks; ++c) {
    if (P.kvb && P.det) {
      for (const char* s : kChunkKvbDetHead) put(s);
      for (int r = 0; r < P.bs; ++r) put("kvb");   // one launch per start residue
      put("dqb");
    } else if (P.det) {
      for (const char* s : kChunkDet) put(s);
    } else if (P.kvb) {
      for (const char* s : kChunkKvb) put(s);
    } else {
      for (const char* s : kChunkKvq) put(s);
    }
  }
  put("cast");
  return n;
}

int64_t launch_count(const Plan& P) { return plan_names(P, nullptr, 0); }

// Host-to-device copies of one chunk's query-side rows (q, qRope, indices,
// softmaxMax, softmaxSum, dOut, out) on the h2d stream, then in_ready[c].
struct HostCopies {
  cudaStream_t h2d;
  const int* bounds;
  const cudaEvent_t* in_ready;
  uint8_t* dq_;   // device copies: q, qRope, indices, max, sum, dO, out
  uint8_t* dqr_;
  uint8_t* didx;
  uint8_t* dmax;
  uint8_t* dsum_;
  uint8_t* ddo;
  uint8_t* dout;
  const uint8_t *hq, *hqr, *hidx, *hmax, *hsum, *hdo, *hout;
  size_t row, rrow, irow, srow;   // bytes per token
  cudaError_t put(int c) const {
    const size_t t0 = c > 0 ? (size_t)bounds[c - 1] : 0, n = (size_t)bounds[c] - t0;
    const cudaMemcpyKind k = cudaMemcpyHostToDevice;
    cudaError_t e = cudaMemcpyAsync(dq_ + t0 * row, hq + t0 * row, n * row, k, h2d);
    if (e == cudaSuccess && rrow) e = cudaMemcpyAsync(dqr_ + t0 * rrow, hqr + t0 * rrow, n * rrow, k, h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(didx + t0 * irow, hidx + t0 * irow, n * irow, k, h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dmax + t0 * srow, hmax + t0 * srow, n * srow, k, h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dsum_ + t0 * srow, hsum + t0 * srow, n * srow, k, h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ddo + t0 * row, hdo + t0 * row, n * row, k, h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dout + t0 * row, hout + t0 * row, n * row, k, h2d);
    if (e == cudaSuccess) e = cudaEventRecord(in_ready[c], h2d);
    return e;
  }
};

// Copy pipeline of sfa_grad_host around the chunk loop.  Before chunk c's
// kernels are queued, chunk c + 1's copies are (so the host queues the first
// kernels after two chunks' copies, not after all of them, and the h2d
// stream still runs one chunk ahead); the compute stream waits for
// in_ready[c] before the chunk's first kernel, and once the chunk's dQ rows
// are final the d2h stream copies them to the host while the next chunk
// computes.
struct Pipe {
  const int* bounds;   // end token of each chunk
  int nch;
  const HostCopies* copies;
  cudaStream_t d2h;
  const cudaEvent_t* in_ready;
  const cudaEvent_t* out_ready;
  void* h_dq;
  void* h_dqr;
};

template <typename T>
sfa_status run_grad(const Plan& P, const sfa_params* prm, const void* q, const void* k, const void* v,
                    const int32_t* idx, const void* dO, const void* out, const float* smax, const float* ssum,
                    const int32_t* aq, const int32_t* akv, const void* qr, const void* kr, void* dq, void* dk, void* dv,
                    void* dqr, void* dkr, uint8_t* ws, cudaStream_t st, Marks mk, const Pipe* pipe = nullptr) {
  int* gerr = reinterpret_cast<int*>(ws + P.off_err);
  Prob pr = make_prob(P, ws);
  pr.q = q; pr.k = k; pr.v = v; pr.dO = dO; pr.out = out; pr.idx = idx;
  pr.qr = P.has_rope ? qr : nullptr;
  pr.kr = P.has_rope ? kr : nullptr;
  pr.smax = smax; pr.ssum = ssum;
  pr.dsum = reinterpret_cast<const float*>(ws + P.off_dsum);
  const int nsm = sm_count();
  Maps maps;
  BlkMaps bmaps;
  if (!make_maps(&maps, P, q, pr.qr, dO, k, pr.kr, v, ws + P.off_P, ws + P.off_dS, dq, P.has_rope ? dqr : nullptr,
                 P.det && !P.kvb ? ws + P.off_part : nullptr) ||
      (P.kvb && !make_blk_maps(&bmaps, P, q, pr.qr, dO, ws + P.off_P, ws + P.off_dS))) {
    snprintf(g_last_error, sizeof(g_last_error), "tensor map encoding failed");
    return SFA_ERR_RUNTIME;
  }
  SFA_CK(mk.mark(st));
  SFA_CK(cudaMemsetAsync(gerr, 0, 16, st));
  SFA_CK(cudaMemsetAsync(ws + P.off_acc, 0, (size_t)P.T2 * kAccRow * 4, st));
  if (P.layout == SFA_LAYOUT_TND) {
    SFA_CK(launch_batch_prefix(pr, P.B, aq, akv, reinterpret_cast<int*>(ws + P.off_batch), gerr, st));
    SFA_CK(mk.mark(st));
  }
  SFA_CK(launch_meta(pr, P.layout, P.B, P.S1, P.S2, P.mode, aq, akv, reinterpret_cast<int*>(ws + P.off_batch),
                     reinterpret_cast<TokMeta*>(ws + P.off_meta), gerr, st));
  SFA_CK(mk.mark(st));
  float* dsum = reinterpret_cast<float*>(ws + P.off_dsum);
  if (!pipe) {
    SFA_CK(launch_dsum<T>(pr, 0, P.T1, dsum, st));
    SFA_CK(mk.mark(st));
  }
  float* acc = reinterpret_cast<float*>(ws + P.off_acc);
  const int nchunks = pipe ? pipe->nch : (P.T1 + P.chunk - 1) / P.chunk;
  for (int c = 0; c < nchunks; ++c) {
    const int t0 = pipe ? (c > 0 ? pipe->bounds[c - 1] : 0) : c * P.chunk;
    const int t_end = pipe ? pipe->bounds[c] : (P.T1 - t0 < P.chunk ? P.T1 : t0 + P.chunk);
    pr.tok0 = t0;
    pr.ntok = t_end - t0;
    if (pipe) {
      if (c + 1 < pipe->nch) SFA_CK(pipe->copies->put(c + 1));
      SFA_CK(cudaStreamWaitEvent(st, pipe->in_ready[c], 0));
      SFA_CK(launch_dsum<T>(pr, t0, pr.ntok, dsum, st));
    }
    void* Pst = ws + P.off_P;
    void* dSst = ws + P.off_dS;
    if (!P.kvb) {   // block indices that many tokens select: no row table, scores per block below
      SFA_CK(launch_rowtab(pr, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_sdp<T>(maps, pr, kModeBwd, nullptr, gerr, nsm, st));
      SFA_CK(mk.mark(st));
    }
    if (P.det && !P.kvb) {
      int* bcnt = reinterpret_cast<int*>(ws + P.off_bcnt);
      int* bcur = reinterpret_cast<int*>(ws + P.off_bcur);
      int* bgrp = reinterpret_cast<int*>(ws + P.off_bgrp);
      int* bbeg = reinterpret_cast<int*>(ws + P.off_bbeg);
      int* bng = reinterpret_cast<int*>(ws + P.off_bng);
      int* bent = reinterpret_cast<int*>(ws + P.off_bent);
      int* dscr = reinterpret_cast<int*>(ws + P.off_dscr);
      uint16_t* part = reinterpret_cast<uint16_t*>(ws + P.off_part);
      SFA_CK(launch_det_count(pr, bcnt, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_blk_scan(bcnt, P.T2, bcur, bgrp, bbeg, bng, 0, nullptr, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_det_scatter(pr, bcur, bent, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_det_sort(pr, bbeg, bng, bent, dscr, false, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_det_sort(pr, bbeg, bng, bent, dscr, true, st));
      SFA_CK(mk.mark(st));
      // key side as partial rows (token-major items) with the query side
      // in the same launch, then the fixed-order sums
      SFA_CK(launch_kvq<T>(maps, pr, reinterpret_cast<float*>(part), dq, P.has_rope ? dqr : nullptr, P.Kpad / 128,
                           true, gerr, nsm, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_det_reduce(pr, bgrp, bbeg, bng, bent, part, acc, st));
      SFA_CK(mk.mark(st));
    } else if (P.kvb) {
      int* bcnt = reinterpret_cast<int*>(ws + P.off_bcnt);
      int* bcur = reinterpret_cast<int*>(ws + P.off_bcur);
      int* bgrp = reinterpret_cast<int*>(ws + P.off_bgrp);
      int* bbeg = reinterpret_cast<int*>(ws + P.off_bbeg);
      int* bng = reinterpret_cast<int*>(ws + P.off_bng);
      int* bent = reinterpret_cast<int*>(ws + P.off_bent);
      SFA_CK(launch_blk_count(pr, bcnt, Pst, dSst, nullptr, st));
      SFA_CK(mk.mark(st));
      int* bres = reinterpret_cast<int*>(ws + P.off_bres);
      SFA_CK(launch_blk_scan(bcnt, P.T2 + P.bs, bcur, bgrp, bbeg, bng, P.bs, bres, st));
      SFA_CK(mk.mark(st));
      SFA_CK(launch_blk_scatter(pr, bcur, bent, st));
      SFA_CK(mk.mark(st));
      if (P.det) {
        // each group's pairs in ascending (token, index) order, so that the
        // tensor-memory accumulation of a block has one fixed order
        SFA_CK(launch_det_sort(pr, bbeg, bng, bent, reinterpret_cast<int*>(ws + P.off_dscr), false, st));
        SFA_CK(mk.mark(st));
        SFA_CK(launch_det_sort(pr, bbeg, bng, bent, reinterpret_cast<int*>(ws + P.off_dscr), true, st));
        SFA_CK(mk.mark(st));
      }
      // scores per block: each block's key / value rows loaded once for all
      // the tokens that select it
      SFA_CK(launch_sdpb<T>(maps, pr, kModeBwd, bgrp, bbeg, bng, bent, Pst, dSst, nullptr, gerr, nsm, st));
      SFA_CK(mk.mark(st));
      if (P.det) {
        // the groups in bs launches by start residue, so that no two tiles
        // added in one launch share a key row
        for (int r = 0; r < P.bs; ++r) {
          SFA_CK(launch_kvb<T>(bmaps, pr, P.bs, bgrp, bbeg, bng, bent, acc, r, bres, gerr, nsm, st));
          SFA_CK(mk.mark(st));
        }
      } else {
        SFA_CK(launch_kvb<T>(bmaps, pr, P.bs, bgrp, bbeg, bng, bent, acc, -1, bres, gerr, nsm, st));
        SFA_CK(mk.mark(st));
      }
      // dQ with the features on the MMA's M (at most 64 heads here)
      SFA_CK(launch_dqb<T>(maps, pr, false, dq, P.has_rope ? dqr : nullptr, nullptr, gerr, nsm, st));
      SFA_CK(mk.mark(st));
    } else {
      SFA_CK(launch_kvq<T>(maps, pr, acc, dq, P.has_rope ? dqr : nullptr, kvq_tile_group(P), false, gerr, nsm, st));
      SFA_CK(mk.mark(st));
    }
    if (pipe) {
      const size_t row = (size_t)P.G * 512 * sizeof(T), rrow = (size_t)P.G * 64 * sizeof(T);
      SFA_CK(cudaEventRecord(pipe->out_ready[c], st));
      SFA_CK(cudaStreamWaitEvent(pipe->d2h, pipe->out_ready[c], 0));
      SFA_CK(cudaMemcpyAsync(static_cast<uint8_t*>(pipe->h_dq) + t0 * row, static_cast<const uint8_t*>(dq) + t0 * row,
                             pr.ntok * row, cudaMemcpyDeviceToHost, pipe->d2h));
      if (P.has_rope)
        SFA_CK(cudaMemcpyAsync(static_cast<uint8_t*>(pipe->h_dqr) + t0 * rrow,
                               static_cast<const uint8_t*>(dqr) + t0 * rrow, pr.ntok * rrow, cudaMemcpyDeviceToHost,
                               pipe->d2h));
    }
  }
  SFA_CK(launch_cast<T>(acc, P.T2, dk, P.has_rope ? dkr : nullptr, dv, P.has_rope, st));
  SFA_CK(mk.mark(st));
  (void)prm;
  return SFA_OK;
}

// Device copies of sfa_grad_host's host buffers, placed after the
// backward's own workspace (byte offsets into the workspace).
struct HostLayout {
  size_t q, k, v, idx, dO, out, smax, ssum, aq, akv, qr, kr, dq, dk, dv, dqr, dkr, total;
};

HostLayout host_layout(const Plan& P) {
  HostLayout L;
  size_t o = P.total;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o += up(bytes);
    return r;
  };
  const size_t t1 = (size_t)P.T1, t2 = (size_t)P.T2, g = (size_t)P.G, e = 2;
  const size_t rope = P.has_rope ? 64 : 0;
  L.q = take(t1 * g * 512 * e);
  L.dO = take(t1 * g * 512 * e);
  L.out = take(t1 * g * 512 * e);
  L.qr = take(t1 * g * rope * e);
  L.idx = take(t1 * (size_t)P.Kidx * 4);
  L.smax = take(t1 * g * 4);
  L.ssum = take(t1 * g * 4);
  L.k = take(t2 * 512 * e);
  L.v = take(t2 * 512 * e);
  L.kr = take(t2 * rope * e);
  L.aq = take((size_t)P.B * 4);
  L.akv = take((size_t)P.B * 4);
  L.dq = take(t1 * g * 512 * e);
  L.dqr = take(t1 * g * rope * e);
  L.dk = take(t2 * 512 * e);
  L.dv = take(t2 * 512 * e);
  L.dkr = take(t2 * rope * e);
  L.total = o;
  return L;
}

// Token chunks of sfa_grad_host (end token of each).  The first chunk is
// small (128 tokens) so that the kernels start after a short copy.  Each
// next chunk is at most `ratio` times larger, where ratio estimates how much
// longer a token's kernels run than its inputs take to copy, so that chunk
// c + 1 lands while chunk c computes.  Chunks stop growing at the staging
// size (cap) and shrink by halves at the end, down to `tmin` tokens, so that
// the last dQ readback is short.
std::vector<int> host_bounds(int T1, int cap, double ratio, int tmin) {
  std::vector<int> b;
  double up = 128.0;
  for (int t = 0; t < T1;) {
    const int rem = T1 - t;
    int n = up < (double)cap ? (int)up : cap;
    const int half = (rem + 1) / 2 > tmin ? (rem + 1) / 2 : tmin;
    if (n > half) n = half;
    if (n > rem) n = rem;
    t += n;
    b.push_back(t);
    up *= ratio;
  }
  return b;
}

// Schedule parameters from the problem shape.  Kernel time per query token
// ~ Kpad x Gp x 9 ps (measured on GB300: MLA 10.3, long context 10.5 ps per
// slot and padded head), or 4 ps on the key-major block plan (block-sparse
// workload 3.9 ps); copy time per token = its input bytes at 200 GB/s
// (pinned host memory measured at 211 GB/s).  The ratio is 0.9 of that
// estimate, kept within [1.25, 8] (causal TND runs slower per slot than the
// estimate, which only makes its ramp cautious).  The tail stops halving at
// the chunk whose dQ readback takes ~0.1 ms at 190 GB/s, and at 128 tokens
// at least.  On MLA the ramp (x1.25) beat even splits into 4, 8 or 16 chunks
// and ramps of x1.5 and x1.15; on the block-sparse workload ramps of x2, x4
// and x8 took 21.2, 20.6 and 20.9 ms end to end (the estimate gives x3.7).
void host_schedule(const Plan& P, double* ratio, int* tmin) {
  const double g = P.G, kernel_s = (double)P.Kpad * P.Gp * (P.kvb ? 4e-12 : 9e-12);
  const double copy_s = (g * (3 * 512 + (P.has_rope ? 64 : 0)) * 2 + (double)P.Kidx * 4 + 2 * g * 4) / 200e9;
  double r = 0.9 * kernel_s / copy_s;
  *ratio = r < 1.25 ? 1.25 : r > 8.0 ? 8.0 : r;
  const double dq_bytes = g * (512 + (P.has_rope ? 64 : 0)) * 2;
  const double tt = 1e-4 * 190e9 / dq_bytes;
  *tmin = tt < 128.0 ? 128 : tt > 1e6 ? 1000000 : (int)tt;
}

// Streams and events of one sfa_grad_host call.  Destroying them with work
// still queued is allowed (the runtime releases them when the work is done);
// on an early error return the internal streams are drained first, so no
// copy from or to the caller's host buffers is still running when the call
// returns.
struct HostRes {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;
  bool joined = false;
  ~HostRes() {
    if (!joined) {
      if (h2d) cudaStreamSynchronize(h2d);
      if (d2h) cudaStreamSynchronize(d2h);
    }
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
  }
};

template <typename T>
sfa_status run_fwd(const Plan& P, const void* q, const void* k, const void* v, const int32_t* idx, const int32_t* aq,
                   const int32_t* akv, const void* qr, const void* kr, void* out, float* smax, float* ssum, uint8_t* ws,
                   cudaStream_t st) {
  int* gerr = reinterpret_cast<int*>(ws + P.off_err);
  Prob pr = make_prob(P, ws);
  pr.q = q; pr.k = k; pr.v = v; pr.idx = idx;
  pr.qr = P.has_rope ? qr : nullptr;
  pr.kr = P.has_rope ? kr : nullptr;
  pr.smax = smax; pr.ssum = ssum;
  const int nsm = sm_count();
  Maps maps;
  if (!make_maps(&maps, P, q, pr.qr, nullptr, k, pr.kr, v, ws + P.off_P, nullptr, out)) {
    snprintf(g_last_error, sizeof(g_last_error), "tensor map encoding failed");
    return SFA_ERR_RUNTIME;
  }
  SFA_CK(cudaMemsetAsync(gerr, 0, 16, st));
  if (P.layout == SFA_LAYOUT_TND)
    SFA_CK(launch_batch_prefix(pr, P.B, aq, akv, reinterpret_cast<int*>(ws + P.off_batch), gerr, st));
  SFA_CK(launch_meta(pr, P.layout, P.B, P.S1, P.S2, P.mode, aq, akv, reinterpret_cast<int*>(ws + P.off_batch),
                     reinterpret_cast<TokMeta*>(ws + P.off_meta), gerr, st));
  float* ts = reinterpret_cast<float*>(ws + P.off_tstats);
  for (int t0 = 0; t0 < P.T1; t0 += P.chunk) {
    pr.tok0 = t0;
    pr.ntok = (P.T1 - t0) < P.chunk ? (P.T1 - t0) : P.chunk;
    if (P.kvb) {
      // block indices that many tokens select: the pairs grouped by block
      // start, statistics per pair with P staged relative to each pair's max,
      // the final statistics, then O per token (features on M, P rescaled)
      int* bcnt = reinterpret_cast<int*>(ws + P.off_bcnt);
      int* bcur = reinterpret_cast<int*>(ws + P.off_bcur);
      int* bgrp = reinterpret_cast<int*>(ws + P.off_bgrp);
      int* bbeg = reinterpret_cast<int*>(ws + P.off_bbeg);
      int* bng = reinterpret_cast<int*>(ws + P.off_bng);
      int* bent = reinterpret_cast<int*>(ws + P.off_bent);
      SFA_CK(launch_blk_count(pr, bcnt, ws + P.off_P, nullptr, ts, st));
      SFA_CK(launch_blk_scan(bcnt, P.T2 + P.bs, bcur, bgrp, bbeg, bng, P.bs, nullptr, st));
      SFA_CK(launch_blk_scatter(pr, bcur, bent, st));
      SFA_CK(launch_sdpb<T>(maps, pr, kModeFwdStats, bgrp, bbeg, bng, bent, ws + P.off_P, nullptr, ts, gerr, nsm, st));
      SFA_CK(launch_stats_combine(pr, ts, P.Kidx, smax, ssum, st));
      SFA_CK(launch_dqb<T>(maps, pr, true, out, nullptr, ts, gerr, nsm, st));
    } else {
      // statistics per 32 slots with P staged relative to each group's max,
      // the final statistics, then O = P V (P rescaled per group)
      SFA_CK(launch_rowtab(pr, st));
      SFA_CK(launch_sdp<T>(maps, pr, kModeFwdStats, ts, gerr, nsm, st));
      SFA_CK(launch_stats_combine(pr, ts, P.Kpad / 32, smax, ssum, st));
      SFA_CK(launch_pv<T>(maps, pr, ts, out, gerr, nsm, st));
    }
  }
  return SFA_OK;
}

}  // namespace
}  // namespace sfa

using sfa::Plan;

extern "C" {

sfa_status sfa_grad_workspace_size(const sfa_params* p, size_t* bytes) {
  if (!p || !bytes) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  *bytes = P.total;
  return SFA_OK;
}

sfa_status sfa_fwd_workspace_size(const sfa_params* p, size_t* bytes) {
  if (!p || !bytes) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, true, &P);
  if (s != SFA_OK) return s;
  *bytes = P.total;
  return SFA_OK;
}

sfa_status sfa_grad(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                    const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                    const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                    void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return sfa_grad_profile(p, q, k, v, indices, d_out, out, softmax_max, softmax_sum, act_seq_q, act_seq_kv, q_rope,
                          k_rope, dq, dk, dv, dq_rope, dk_rope, workspace, workspace_bytes, stream, nullptr, 0);
}

sfa_status sfa_grad_plan_info(const sfa_params* p, int64_t* chunk_tokens, int64_t* kernel_launches) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  if (chunk_tokens) *chunk_tokens = P.chunk;
  if (kernel_launches) *kernel_launches = P.T1 == 0 ? 0 : sfa::launch_count(P);
  return SFA_OK;
}

sfa_status sfa_grad_plan_names(const sfa_params* p, const char** names, int32_t capacity, int32_t* count) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  const int64_t n = sfa::plan_names(P, names, capacity > 0 ? capacity : 0);
  if (count) *count = (int32_t)n;
  return SFA_OK;
}

sfa_status sfa_grad_profile(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                            const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                            const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope,
                            const void* k_rope, void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope,
                            void* workspace, size_t workspace_bytes, void* stream, void** events, int32_t n_events) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool rope = P.has_rope;
  if (!dk || !dv || (rope && !dk_rope)) return SFA_ERR_NULLPTR;
  if (P.T1 == 0) {  // empty query: nothing selects any key
    if (P.T2 > 0) {
      const size_t esz = 2;
      SFA_CK(cudaMemsetAsync(dk, 0, (size_t)P.T2 * 512 * esz, st));
      SFA_CK(cudaMemsetAsync(dv, 0, (size_t)P.T2 * 512 * esz, st));
      if (rope) SFA_CK(cudaMemsetAsync(dk_rope, 0, (size_t)P.T2 * 64 * esz, st));
    }
    return SFA_OK;
  }
  if (!q || !k || !v || !indices || !d_out || !out || !softmax_max || !softmax_sum || !dq || !workspace)
    return SFA_ERR_NULLPTR;
  if (rope && (!q_rope || !k_rope || !dq_rope)) return SFA_ERR_NULLPTR;
  if (P.layout == SFA_LAYOUT_TND && (!act_seq_q || !act_seq_kv)) return SFA_ERR_NULLPTR;
  if (workspace_bytes < P.total) return SFA_ERR_PARAM_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sfa::Marks mk;
  mk.ev = events;
  mk.n = events ? n_events : 0;
  if (P.is_f16)
    return sfa::run_grad<__half>(P, p, q, k, v, indices, d_out, out, softmax_max, softmax_sum, act_seq_q, act_seq_kv,
                                 q_rope, k_rope, dq, dk, dv, dq_rope, dk_rope, ws, st, mk);
  return sfa::run_grad<__nv_bfloat16>(P, p, q, k, v, indices, d_out, out, softmax_max, softmax_sum, act_seq_q,
                                      act_seq_kv, q_rope, k_rope, dq, dk, dv, dq_rope, dk_rope, ws, st, mk);
}

sfa_status sfa_grad_host_workspace_size(const sfa_params* p, size_t* bytes) {
  if (!p || !bytes) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  *bytes = sfa::host_layout(P).total;
  return SFA_OK;
}

sfa_status sfa_grad_host(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                         const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                         const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                         void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  const sfa::HostLayout L = sfa::host_layout(P);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool rope = P.has_rope;
  if (!dk || !dv || (rope && !dk_rope) || !workspace) return SFA_ERR_NULLPTR;
  if (workspace_bytes < L.total) return SFA_ERR_PARAM_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t e = 2, t2 = (size_t)P.T2, g = (size_t)P.G;
  const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
  if (P.T1 == 0) {  // empty query: nothing selects any key
    if (P.T2 > 0) {
      SFA_CK(cudaMemsetAsync(ws + L.dk, 0, L.total - L.dk, st));   // dk, dv, dkr
      SFA_CK(cudaMemcpyAsync(dk, ws + L.dk, t2 * 512 * e, D2H, st));
      SFA_CK(cudaMemcpyAsync(dv, ws + L.dv, t2 * 512 * e, D2H, st));
      if (rope) SFA_CK(cudaMemcpyAsync(dk_rope, ws + L.dkr, t2 * 64 * e, D2H, st));
    }
    return SFA_OK;
  }
  if (!q || !k || !v || !indices || !d_out || !out || !softmax_max || !softmax_sum || !dq) return SFA_ERR_NULLPTR;
  if (rope && (!q_rope || !k_rope || !dq_rope)) return SFA_ERR_NULLPTR;
  if (P.layout == SFA_LAYOUT_TND && (!act_seq_q || !act_seq_kv)) return SFA_ERR_NULLPTR;
  const bool shared_kv = v == k;
  double ratio;
  int tmin;
  sfa::host_schedule(P, &ratio, &tmin);
  const std::vector<int> bounds = sfa::host_bounds(P.T1, P.chunk, ratio, tmin);
  const int nch = (int)bounds.size();

  sfa::HostRes R;
  SFA_CK(cudaStreamCreateWithFlags(&R.h2d, cudaStreamNonBlocking));
  SFA_CK(cudaStreamCreateWithFlags(&R.d2h, cudaStreamNonBlocking));
  R.ev.reserve(4 + 2 * (size_t)nch);
  for (int i = 0; i < 4 + 2 * nch; ++i) {
    cudaEvent_t ev;
    SFA_CK(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    R.ev.push_back(ev);
  }
  const cudaEvent_t ev_start = R.ev[0], ev_kv = R.ev[1], ev_cast = R.ev[2], ev_done = R.ev[3];
  const cudaEvent_t* in_ready = R.ev.data() + 4;
  const cudaEvent_t* out_ready = R.ev.data() + 4 + nch;

  // the copies start once earlier work on the caller's stream (which may
  // still read this workspace) is done
  SFA_CK(cudaEventRecord(ev_start, st));
  SFA_CK(cudaStreamWaitEvent(R.h2d, ev_start, 0));
  SFA_CK(cudaMemcpyAsync(ws + L.k, k, t2 * 512 * e, H2D, R.h2d));
  if (!shared_kv) SFA_CK(cudaMemcpyAsync(ws + L.v, v, t2 * 512 * e, H2D, R.h2d));
  if (rope) SFA_CK(cudaMemcpyAsync(ws + L.kr, k_rope, t2 * 64 * e, H2D, R.h2d));
  if (P.layout == SFA_LAYOUT_TND) {
    SFA_CK(cudaMemcpyAsync(ws + L.aq, act_seq_q, (size_t)P.B * 4, H2D, R.h2d));
    SFA_CK(cudaMemcpyAsync(ws + L.akv, act_seq_kv, (size_t)P.B * 4, H2D, R.h2d));
  }
  SFA_CK(cudaEventRecord(ev_kv, R.h2d));
  // the first chunk's query-side rows; run_grad queues each next chunk's
  // before the current chunk's kernels
  sfa::HostCopies hc;
  hc.h2d = R.h2d;
  hc.bounds = bounds.data();
  hc.in_ready = in_ready;
  hc.dq_ = ws + L.q;
  hc.dqr_ = ws + L.qr;
  hc.didx = ws + L.idx;
  hc.dmax = ws + L.smax;
  hc.dsum_ = ws + L.ssum;
  hc.ddo = ws + L.dO;
  hc.dout = ws + L.out;
  hc.hq = static_cast<const uint8_t*>(q);
  hc.hqr = static_cast<const uint8_t*>(q_rope);
  hc.hidx = reinterpret_cast<const uint8_t*>(indices);
  hc.hmax = reinterpret_cast<const uint8_t*>(softmax_max);
  hc.hsum = reinterpret_cast<const uint8_t*>(softmax_sum);
  hc.hdo = static_cast<const uint8_t*>(d_out);
  hc.hout = static_cast<const uint8_t*>(out);
  hc.row = g * 512 * e;
  hc.rrow = rope ? g * 64 * e : 0;
  hc.irow = (size_t)P.Kidx * 4;
  hc.srow = g * 4;
  SFA_CK(hc.put(0));

  SFA_CK(cudaStreamWaitEvent(st, ev_kv, 0));
  sfa::Pipe pipe;
  pipe.bounds = bounds.data();
  pipe.nch = nch;
  pipe.copies = &hc;
  pipe.d2h = R.d2h;
  pipe.in_ready = in_ready;
  pipe.out_ready = out_ready;
  pipe.h_dq = dq;
  pipe.h_dqr = dq_rope;
  uint8_t* d_v = shared_kv ? ws + L.k : ws + L.v;
  const int32_t* d_aq = P.layout == SFA_LAYOUT_TND ? reinterpret_cast<const int32_t*>(ws + L.aq) : nullptr;
  const int32_t* d_akv = P.layout == SFA_LAYOUT_TND ? reinterpret_cast<const int32_t*>(ws + L.akv) : nullptr;
  if (P.is_f16)
    s = sfa::run_grad<__half>(P, p, ws + L.q, ws + L.k, d_v, reinterpret_cast<const int32_t*>(ws + L.idx), ws + L.dO,
                              ws + L.out, reinterpret_cast<const float*>(ws + L.smax),
                              reinterpret_cast<const float*>(ws + L.ssum), d_aq, d_akv, ws + L.qr, ws + L.kr,
                              ws + L.dq, ws + L.dk, ws + L.dv, ws + L.dqr, ws + L.dkr, ws, st, sfa::Marks{}, &pipe);
  else
    s = sfa::run_grad<__nv_bfloat16>(P, p, ws + L.q, ws + L.k, d_v, reinterpret_cast<const int32_t*>(ws + L.idx),
                                     ws + L.dO, ws + L.out, reinterpret_cast<const float*>(ws + L.smax),
                                     reinterpret_cast<const float*>(ws + L.ssum), d_aq, d_akv, ws + L.qr, ws + L.kr,
                                     ws + L.dq, ws + L.dk, ws + L.dv, ws + L.dqr, ws + L.dkr, ws, st, sfa::Marks{},
                                     &pipe);
  if (s != SFA_OK) return s;
  // key-side outputs after the final cast, then the caller's stream waits
  // for every copy to the host
  SFA_CK(cudaEventRecord(ev_cast, st));
  SFA_CK(cudaStreamWaitEvent(R.d2h, ev_cast, 0));
  SFA_CK(cudaMemcpyAsync(dk, ws + L.dk, t2 * 512 * e, D2H, R.d2h));
  SFA_CK(cudaMemcpyAsync(dv, ws + L.dv, t2 * 512 * e, D2H, R.d2h));
  if (rope) SFA_CK(cudaMemcpyAsync(dk_rope, ws + L.dkr, t2 * 64 * e, D2H, R.d2h));
  SFA_CK(cudaEventRecord(ev_done, R.d2h));
  SFA_CK(cudaStreamWaitEvent(st, ev_done, 0));
  R.joined = true;
  return SFA_OK;
}

sfa_status sfa_fwd(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                   const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                   void* out, float* softmax_max, float* softmax_sum, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, true, &P);
  if (s != SFA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (P.T1 == 0) return SFA_OK;
  if (!q || !k || !v || !indices || !out || !softmax_max || !softmax_sum || !workspace) return SFA_ERR_NULLPTR;
  if (P.has_rope && (!q_rope || !k_rope)) return SFA_ERR_NULLPTR;
  if (P.layout == SFA_LAYOUT_TND && (!act_seq_q || !act_seq_kv)) return SFA_ERR_NULLPTR;
  if (workspace_bytes < P.total) return SFA_ERR_PARAM_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (P.is_f16)
    return sfa::run_fwd<__half>(P, q, k, v, indices, act_seq_q, act_seq_kv, q_rope, k_rope, out, softmax_max,
                                softmax_sum, ws, st);
  return sfa::run_fwd<__nv_bfloat16>(P, q, k, v, indices, act_seq_q, act_seq_kv, q_rope, k_rope, out, softmax_max,
                                     softmax_sum, ws, st);
}

sfa_status sfa_decode_keys(const sfa_params* p, const int32_t* indices, const int32_t* act_seq_q,
                           const int32_t* act_seq_kv, int32_t* rows_out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!p) return SFA_ERR_NULLPTR;
  Plan P;
  sfa_status s = sfa::validate(p, false, &P);
  if (s != SFA_OK) return s;
  if (P.T1 == 0) return SFA_OK;
  if (!indices || !rows_out || !workspace) return SFA_ERR_NULLPTR;
  if (P.layout == SFA_LAYOUT_TND && (!act_seq_q || !act_seq_kv)) return SFA_ERR_NULLPTR;
  if (workspace_bytes < P.total) return SFA_ERR_PARAM_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* gerr = reinterpret_cast<int*>(ws + P.off_err);
  sfa::Prob pr = sfa::make_prob(P, ws);
  pr.idx = indices;
  SFA_CK(cudaMemsetAsync(gerr, 0, 16, st));
  if (P.layout == SFA_LAYOUT_TND)
    SFA_CK(sfa::launch_batch_prefix(pr, P.B, act_seq_q, act_seq_kv, reinterpret_cast<int*>(ws + P.off_batch), gerr, st));
  SFA_CK(sfa::launch_meta(pr, P.layout, P.B, P.S1, P.S2, P.mode, act_seq_q, act_seq_kv,
                          reinterpret_cast<int*>(ws + P.off_batch), reinterpret_cast<sfa::TokMeta*>(ws + P.off_meta),
                          gerr, st));
  sfa::decode_kernel<<<1024, 256, 0, st>>>(pr, rows_out);
  SFA_CK(cudaGetLastError());
  return SFA_OK;
}

sfa_status sfa_read_device_error(void* workspace, void* stream, int32_t* code) {
  if (!workspace || !code) return SFA_ERR_NULLPTR;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  SFA_CK(cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st));
  SFA_CK(cudaStreamSynchronize(st));
  SFA_CK(cudaMemsetAsync(workspace, 0, 4, st));
  *code = v;
  return SFA_OK;
}

const char* sfa_last_error_message(void) { return sfa::g_last_error; }

const char* sfa_status_string(int32_t s) {
  switch (s) {
    case SFA_OK: return "SFA_OK";
    case SFA_ERR_NULLPTR: return "SFA_ERR_NULLPTR: a required pointer is null";
    case SFA_ERR_PARAM_INVALID: return "SFA_ERR_PARAM_INVALID: dtype/layout out of range or workspace too small";
    case SFA_ERR_RUNTIME: return "SFA_ERR_RUNTIME: a CUDA call failed";
    case SFA_ERR_SHAPE: return "SFA_ERR_SHAPE: size or attribute outside the supported range";
    default: return "unknown sfa status";
  }
}

}  // extern "C"
