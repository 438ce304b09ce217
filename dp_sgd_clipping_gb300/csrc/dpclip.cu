// C-ABI of libdpclip: argument checks, workspace layout, TMA tensor maps and
// the launch sequence of each entry point on the caller's stream.
//
// Entry points and the passages they implement (randomized-clipping summary
// = "Technical summary: efficient DP-SGD for LLMs with randomized clipping",
// gist.science; glossary = "DP-SGD" entry of jisaku.com):
//   dpclip_norms_exact         trace identity, "Core mechanism"; ghost and
//                              direct forms of "Problem definition"
//   dpclip_norms_hutch         "Core mechanism", item 1
//   dpclip_norms_hutchpp       "Core mechanism", item 2
//   dpclip_clipped_noisy_grad  glossary "DP-SGD algorithm" steps 3-4;
//                              "Algorithmic flow" steps 4-5
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "internal.h"

namespace dpclip {
namespace {

constexpr size_t kAlign = 256;
constexpr int kTargetCtas = 304;      // two resident CTAs on each of 152 SMs

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// Carves named regions out of the workspace; offsets are 256-byte aligned.
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = align_up(off, kAlign);
    off = o + bytes;
    return o;
  }
  size_t total() const { return align_up(off, kAlign); }
};

// K-split factor of a skinny GEMM: enough CTAs to keep ~two per SM resident,
// at least 4 K-blocks per split, no empty split, at most kMaxSplits (the
// splits of a tile form one cluster).
void choose_splits(int ntiles, int kblocks, int& splits, int& per) {
  int s = std::max(1, kTargetCtas / std::max(1, ntiles));
  s = std::min(s, std::max(1, kblocks / 4));
  s = std::min(s, kMaxSplits);
  per = cdiv(kblocks, s);
  splits = cdiv(kblocks, per);
}

// ------------------------------------------------------------------ TMA maps
using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeFn) nullptr;
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}

// bf16 tensor [n2][n1][n0] (n0 innermost), box {b0, b1, 1}, 128-byte swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* base, long long n0, long long n1, long long n2, int b0,
              int b1) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)n0, (cuuint64_t)n1, (cuuint64_t)n2};
  const cuuint64_t strides[2] = {(cuuint64_t)n0 * 2, (cuuint64_t)n0 * n1 * 2};
  const cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ checks
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shapes(const void* A, const void* G, int B, int T, int d, int p, int dtype) {
  if (!A || !G) return DPCLIP_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || d <= 0 || p <= 0) return DPCLIP_ERR_INVALID_ARG;
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  if ((long long)d * p > (1ll << 34)) return DPCLIP_ERR_UNSUPPORTED;   // Philox block index
  if ((long long)B * T > (1ll << 30)) return DPCLIP_ERR_UNSUPPORTED;
  if (dtype == DPCLIP_BF16) {
    if (d % 8 || p % 8) return DPCLIP_ERR_UNSUPPORTED;   // 16-byte TMA row strides
    if (!aligned(A, 16) || !aligned(G, 16)) return DPCLIP_ERR_UNSUPPORTED;
  } else {
    if (!aligned(A, 4) || !aligned(G, 4)) return DPCLIP_ERR_UNSUPPORTED;
  }
  return DPCLIP_OK;
}

int check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return DPCLIP_ERR_WORKSPACE;
  if (!aligned(ws, kAlign)) return DPCLIP_ERR_WORKSPACE;
  if (ws_bytes < need) return DPCLIP_ERR_WORKSPACE;
  return DPCLIP_OK;
}

int resolve_exact(int method, int T, int d, int p) {
  if (method == DPCLIP_EXACT_AUTO) {
    const double ghost = (double)T * T * (d + p);   // upper triangle of two T x T Grams
    const double direct = 2.0 * T * d * p;
    return direct < ghost ? DPCLIP_EXACT_DIRECT : DPCLIP_EXACT_GHOST;
  }
  return method;
}

// ------------------------------------------------------------------ plans
// Every workspace starts with a control block: word 0 = device error code,
// then the integer tickets of the split reductions.  It is cleared at the
// start of each call.
struct Plan {
  size_t total = 0;
  size_t ctrl = 0, ctrl_bytes = 0;
  size_t off[16] = {};
  // skinny-GEMM geometry
  int mtiles = 0, Tp = 0, tblocks = 0;
};

enum {
  kP = 0, kYhi, kYlo, kQpart,                                // hutch
  kS = 0, kGp, kY1hi, kY1lo, kZ1hi, kZ1lo, kUhi, kUlo,       // hutch++ ...
  kV, kQWhi, kQWlo, kY3hi, kY3lo, kHQpart,
};

int np_for(int n) { return n <= 16 ? 16 : 32; }

Plan plan_hutch_bf16(int B, int T, int d, int p, int k) {
  Plan pl;
  const int NP = np_for(k);
  pl.mtiles = cdiv(T, kTokTileM);
  pl.Tp = pl.mtiles * kTokTileM;
  pl.tblocks = cdiv(T, kBlockK);
  const int ftiles = cdiv(d, kFeatTileM);
  Carve c;
  pl.ctrl_bytes = align_up(4 * (1 + (size_t)B), kAlign);   // error word, per-sample tickets
  pl.ctrl = c.take(pl.ctrl_bytes);
  pl.off[kP] = c.take((size_t)NP * p * 2);
  pl.off[kYhi] = c.take((size_t)B * NP * pl.Tp * 2);
  pl.off[kYlo] = c.take((size_t)B * NP * pl.Tp * 2);
  pl.off[kQpart] = c.take((size_t)B * ftiles * kMaxSplits * 4);
  pl.total = c.total();
  return pl;
}

Plan plan_hutchpp_bf16(int B, int T, int d, int p, int k) {
  Plan pl;
  const int r = k / 3, m = k - 2 * r;
  (void)m;
  pl.mtiles = cdiv(T, kTokTileM);
  pl.Tp = pl.mtiles * kTokTileM;
  pl.tblocks = cdiv(T, kBlockK);
  const int fd = cdiv(d, kFeatTileM), fp = cdiv(p, kFeatTileM);
  Carve c;
  pl.ctrl_bytes = align_up(4 * (1 + (size_t)B), kAlign);   // error word, per-sample tickets
  pl.ctrl = c.take(pl.ctrl_bytes);
  pl.off[kS] = c.take((size_t)16 * p * 2);
  pl.off[kGp] = c.take((size_t)32 * p * 2);
  pl.off[kY1hi] = c.take((size_t)B * 16 * pl.Tp * 2);
  pl.off[kY1lo] = c.take((size_t)B * 16 * pl.Tp * 2);
  pl.off[kZ1hi] = c.take((size_t)B * 16 * d * 2);
  pl.off[kZ1lo] = c.take((size_t)B * 16 * d * 2);
  pl.off[kUhi] = c.take((size_t)B * 16 * pl.Tp * 2);
  pl.off[kUlo] = c.take((size_t)B * 16 * pl.Tp * 2);
  pl.off[kV] = c.take((size_t)B * 16 * p * 4);
  pl.off[kQWhi] = c.take((size_t)B * 32 * p * 2);
  pl.off[kQWlo] = c.take((size_t)B * 32 * p * 2);
  pl.off[kY3hi] = c.take((size_t)B * 32 * pl.Tp * 2);
  pl.off[kY3lo] = c.take((size_t)B * 32 * pl.Tp * 2);
  pl.off[kHQpart] = c.take((size_t)B * std::max(fd, fp) * kMaxSplits * 4);
  pl.total = c.total();
  return pl;
}

// CTA tiles of the gradient / direct-norm GEMM (pairs of 128-row tiles).
int dp_mtiles(int d) { return 2 * cdiv(d, 2 * kDpTileM); }
int dp_ntiles(int d, int p) { return dp_mtiles(d) * cdiv(p, kDpTileN); }
// ghost units per sample: the 256-token tile pairs a' <= b'.
int ghost_npairs(int T) {
  const int n = cdiv(T, 2 * kGhostTile);
  return n * (n + 1) / 2;
}

Plan plan_exact_bf16(int B, int T, int d, int p, int method) {
  Plan pl;
  Carve c;
  const bool ghost = method != DPCLIP_EXACT_DIRECT;
  const size_t xunits = std::min<size_t>(kGhostSharedUnits, (size_t)ghost_npairs(T) * B);
  // error word, grid ticket; ghost: the ready counters of a shared X (one
  // per unit, CTA rank and epilogue warp)
  pl.ctrl_bytes = ghost ? align_up(4 * (2 + xunits * 2 * kEpiWarps), kAlign) : kAlign;
  pl.ctrl = c.take(pl.ctrl_bytes);
  // direct: one partial per CTA tile, sample and epilogue warp.  ghost: whole
  // units plus at most 8 sub-units for each unit of the last round (fewer
  // than one per pair), two CTAs x kEpiWarps partials each
  const size_t parts =
      method == DPCLIP_EXACT_DIRECT
          ? (size_t)dp_ntiles(d, p) * B * kEpiWarps
          : ((size_t)ghost_npairs(T) * B + 8 * (size_t)(kMaxPersistentGrid / 2)) * 2 * kEpiWarps;
  pl.off[0] = c.take(parts * 4);
  if (ghost) pl.off[1] = c.take(xunits * 2 * 128 * 256 * 4);   // shared X of the last round
  pl.total = c.total();
  return pl;
}

// fp32 plans
enum { kFP = 0, kFY, kFPart, kFS, kFGp, kFY1, kFZ1, kFU, kFV, kFQW, kFY3, kFW };

Plan plan_hutch_f32(int B, int T, int d, int p, int k) {
  Plan pl;
  Carve c;
  pl.ctrl_bytes = kAlign;
  pl.ctrl = c.take(pl.ctrl_bytes);
  pl.off[kFP] = c.take((size_t)k * p * 4);
  pl.off[kFY] = c.take((size_t)B * T * k * 4);
  pl.off[kFPart] = c.take((size_t)B * simt_nblocks(d, k) * 4);
  pl.total = c.total();
  return pl;
}

Plan plan_hutchpp_f32(int B, int T, int d, int p, int k) {
  Plan pl;
  const int r = k / 3, m = k - 2 * r;
  Carve c;
  pl.ctrl_bytes = kAlign;
  pl.ctrl = c.take(pl.ctrl_bytes);
  pl.off[kFS] = c.take((size_t)r * p * 4);
  pl.off[kFGp] = c.take((size_t)m * p * 4);
  pl.off[kFY1] = c.take((size_t)B * T * r * 4);
  pl.off[kFZ1] = c.take((size_t)B * d * r * 4);
  pl.off[kFU] = c.take((size_t)B * T * r * 4);
  pl.off[kFV] = c.take((size_t)B * 16 * p * 4);
  pl.off[kFQW] = c.take((size_t)B * 32 * p * 4);
  pl.off[kFY3] = c.take((size_t)B * T * (r + m) * 4);
  pl.off[kFPart] = c.take((size_t)B * simt_nblocks(d, r + m) * 4);
  pl.total = c.total();
  return pl;
}

Plan plan_exact_f32(int B, int T, int d, int p, int method) {
  Plan pl;
  Carve c;
  pl.ctrl_bytes = kAlign;
  pl.ctrl = c.take(pl.ctrl_bytes);
  if (method == DPCLIP_EXACT_DIRECT) {
    pl.off[kFPart] = c.take((size_t)B * simt_nblocks(d, p) * 4);
  } else {
    pl.off[kFW] = c.take((size_t)B * T * T * 4);
    pl.off[kFPart] = c.take((size_t)B * simt_nblocks(T, T) * 4);
  }
  pl.total = c.total();
  return pl;
}

// Gradient: tile tickets in the control block, plus the partial-tile slots of
// the balanced tail (bf16 only).
Plan plan_grad(int d, int p, int dtype) {
  Plan pl;
  Carve c;
  if (dtype == DPCLIP_BF16) {
    pl.ctrl_bytes = align_up(4 * (1 + (size_t)dp_ntiles(d, p)), kAlign);
    pl.ctrl = c.take(pl.ctrl_bytes);
    pl.off[0] = c.take(gemm_dp_slot_bytes(kMaxPersistentGrid));
  } else {
    pl.ctrl_bytes = kAlign;
    pl.ctrl = c.take(pl.ctrl_bytes);
  }
  pl.total = c.total();
  return pl;
}

// Stored direct norms: the control block, then the per-sample gradients M
// (at offset kAlign, so that the gradient call finds them from B, d and p
// alone; sample i at i * stored_stride floats), then the norm partials.
constexpr int kStoredSqBlocks = 64;   // fp32 path: chunks per sample of ||M_i||^2
size_t stored_stride(int d, int p) { return ((size_t)d * p + 3) / 4 * 4; }

Plan plan_stored(int B, int d, int p, int dtype) {
  Plan pl;
  Carve c;
  pl.ctrl_bytes = kAlign;
  pl.ctrl = c.take(pl.ctrl_bytes);
  pl.off[0] = c.take((size_t)B * stored_stride(d, p) * 4);
  pl.off[1] = c.take(dtype == DPCLIP_BF16 ? (size_t)dp_ntiles(d, p) * B * kEpiWarps * 4
                                          : (size_t)B * kStoredSqBlocks * 4);
  pl.total = c.total();
  return pl;
}

int hutch_k_ok(int k) { return k >= 1 && k <= DPCLIP_HUTCH_MAX_K; }
int hutchpp_k_ok(int k) { return k >= 3 && k <= DPCLIP_HUTCHPP_MAX_K && (k - k / 3) <= kMaxNP; }

int plan_for(int op, int B, int T, int d, int p, int dtype, int param, Plan& pl) {
  switch (op) {
    case DPCLIP_OP_NORMS_EXACT: {
      if (param < DPCLIP_EXACT_AUTO || param > DPCLIP_EXACT_DIRECT) return DPCLIP_ERR_INVALID_ARG;
      const int m = resolve_exact(param, T, d, p);
      pl = dtype == DPCLIP_BF16 ? plan_exact_bf16(B, T, d, p, m) : plan_exact_f32(B, T, d, p, m);
      return DPCLIP_OK;
    }
    case DPCLIP_OP_NORMS_HUTCH:
      if (!hutch_k_ok(param)) return DPCLIP_ERR_UNSUPPORTED;
      pl = dtype == DPCLIP_BF16 ? plan_hutch_bf16(B, T, d, p, param) : plan_hutch_f32(B, T, d, p, param);
      return DPCLIP_OK;
    case DPCLIP_OP_NORMS_HUTCHPP:
      if (!hutchpp_k_ok(param)) return DPCLIP_ERR_UNSUPPORTED;
      pl = dtype == DPCLIP_BF16 ? plan_hutchpp_bf16(B, T, d, p, param)
                                : plan_hutchpp_f32(B, T, d, p, param);
      return DPCLIP_OK;
    case DPCLIP_OP_CLIPPED_NOISY_GRAD:
      pl = plan_grad(d, p, dtype);
      return DPCLIP_OK;
    case DPCLIP_OP_STORED_DIRECT:
      pl = plan_stored(B, d, p, dtype);
      return DPCLIP_OK;
    case DPCLIP_OP_BIAS: {
      Carve c;
      pl.ctrl_bytes = 0;
      pl.off[0] = c.take(bias_part_floats(B, T, p) * 4);
      pl.total = c.total();
      return DPCLIP_OK;
    }
    default:
      return DPCLIP_ERR_INVALID_ARG;
  }
}

#define DPCLIP_CUDA(call)                        \
  do {                                           \
    if ((call) != cudaSuccess) {                 \
      (void)cudaGetLastError();                  \
      return DPCLIP_ERR_CUDA;                    \
    }                                            \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Hutch++'s second pass over G (feature-side, each CTA walking its tokens in
// order) leaves the last tokens' rows of G in L2 for the third pass when it
// loads them with the default policy instead of evict-first: as many 64-token
// blocks as fit in L2 beside A with a 24 MB margin (12 MB measured the same,
// 40 MB half as good).  Returns the first kept token.
int hpp_keep_t0(int B, int T, int d, int p) {
  static int l2 = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      v = 0;
    return v;
  }();
  const double a_bytes = 2.0 * B * T * (double)d;
  const double room = (double)l2 - a_bytes - 24e6;
  if (room <= 0) return 1 << 30;
  const double per_block = 2.0 * B * kBlockK * (double)p;   // one 64-token block of every sample
  const int blocks = (int)std::min<double>(room / per_block, (double)cdiv(T, kBlockK));
  return blocks <= 0 ? (1 << 30) : std::max(0, T - blocks * kBlockK);
}

// ------------------------------------------------------------------ skinny launches
int run_tok(const void* X, int B, int T, int F, const void* Whi, const void* Wlo, int NP,
            bool per_sample, const Plan& pl, void* ws, void* out_hi, void* out_lo,
            cudaStream_t s, bool x_stream = false) {
  TokGemmParams tp;
  std::memset(&tp, 0, sizeof(tp));
  const int Bw = per_sample ? B : 1;
  if (!make_map(&tp.map_x, X, F, T, B, kBlockK, kTokTileM)) return DPCLIP_ERR_UNSUPPORTED;
  if (!make_map(&tp.map_whi, Whi, F, NP, Bw, kBlockK, NP)) return DPCLIP_ERR_UNSUPPORTED;
  if (Wlo) {
    if (!make_map(&tp.map_wlo, Wlo, F, NP, Bw, kBlockK, NP)) return DPCLIP_ERR_UNSUPPORTED;
  } else {
    tp.map_wlo = tp.map_whi;
  }
  tp.B = B;
  tp.T = T;
  tp.F = F;
  tp.NP = NP;
  tp.w_per_sample = per_sample ? 1 : 0;
  tp.has_lo = Wlo ? 1 : 0;
  tp.mtiles = pl.mtiles;
  tp.kblocks = cdiv(F, kBlockK);
  choose_splits(B * pl.mtiles, tp.kblocks, tp.splits, tp.kb_per_split);
  tp.Tp = pl.Tp;
  tp.x_stream = x_stream ? 1 : 0;
  tp.out_hi = static_cast<__nv_bfloat16*>(out_hi);
  tp.out_lo = static_cast<__nv_bfloat16*>(out_lo);
  tp.err = at<uint32_t>(ws, pl.ctrl);
  DPCLIP_CUDA(launch_tok_gemm(tp, s));
  return DPCLIP_OK;
}

int run_feat(const void* X, int B, int T, int F, const void* Yhi, const void* Ylo, int NP, int mode,
             const float* w, const Plan& pl, void* ws, size_t qpart_off,
             float* out_f32, void* out_hi, void* out_lo, float* sq, cudaStream_t s,
             bool x_stream = false, int x_keep_t0 = 1 << 30) {
  FeatGemmParams fp;
  std::memset(&fp, 0, sizeof(fp));
  if (!make_map(&fp.map_x, X, F, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
  if (!make_map(&fp.map_yhi, Yhi, pl.Tp, NP, B, kBlockK, NP)) return DPCLIP_ERR_UNSUPPORTED;
  if (!make_map(&fp.map_ylo, Ylo, pl.Tp, NP, B, kBlockK, NP)) return DPCLIP_ERR_UNSUPPORTED;
  fp.B = B;
  fp.T = T;
  fp.F = F;
  fp.NP = NP;
  fp.Tp = pl.Tp;
  fp.ftiles = cdiv(F, kFeatTileM);
  fp.Fp = fp.ftiles * kFeatTileM;
  fp.tblocks = pl.tblocks;
  choose_splits(B * fp.ftiles, fp.tblocks, fp.splits, fp.tb_per_split);
  for (int j = 0; j < kMaxNP; ++j) fp.w[j] = w ? w[j] : 0.f;
  fp.out_f32 = out_f32;
  fp.out_hi = static_cast<__nv_bfloat16*>(out_hi);
  fp.out_lo = static_cast<__nv_bfloat16*>(out_lo);
  fp.sq = sq;
  fp.qpart = at<float>(ws, qpart_off);
  fp.counters = at<uint32_t>(ws, pl.ctrl + 4);
  fp.x_stream = x_stream ? 1 : 0;
  fp.x_keep_t0 = x_keep_t0;
  fp.err = at<uint32_t>(ws, pl.ctrl);
  DPCLIP_CUDA(launch_feat_gemm(fp, mode, s));
  return DPCLIP_OK;
}

SimtParams simt_base() {
  SimtParams sp;
  std::memset(&sp, 0, sizeof(sp));
  for (int j = 0; j < 64; ++j) sp.w[j] = 1.f;
  return sp;
}

#define DPCLIP_TRY(expr)           \
  do {                             \
    const int st_ = (expr);        \
    if (st_ != DPCLIP_OK) return st_; \
  } while (0)

}  // namespace
}  // namespace dpclip

using namespace dpclip;

extern "C" {

const char* dpclip_version(void) { return "dpclip 0.1 (sm_103a)"; }

const char* dpclip_status_string(int status) {
  switch (status) {
    case DPCLIP_OK: return "ok";
    case DPCLIP_ERR_INVALID_ARG: return "invalid argument";
    case DPCLIP_ERR_UNSUPPORTED: return "unsupported shape, alignment or parameter";
    case DPCLIP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DPCLIP_ERR_CUDA: return "CUDA error";
    case DPCLIP_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int dpclip_workspace_size(int op, int B, int T, int d, int p, int dtype, int param, size_t* bytes) {
  if (!bytes) return DPCLIP_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || p <= 0 || (d <= 0 && op != DPCLIP_OP_BIAS)) return DPCLIP_ERR_INVALID_ARG;
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  Plan pl;
  DPCLIP_TRY(plan_for(op, B, T, d, p, dtype, param, pl));
  *bytes = pl.total;
  return DPCLIP_OK;
}

int dpclip_philox_normal(void* out, int64_t n, int dtype, uint64_t seed, uint32_t stream_id,
                         uint64_t offset, dpclip_stream_t stream) {
  if (!out || n < 0) return DPCLIP_ERR_INVALID_ARG;
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  if (!aligned(out, 4)) return DPCLIP_ERR_UNSUPPORTED;
  if (n > (int64_t)4 * 0xFFFFFFFFll) return DPCLIP_ERR_UNSUPPORTED;
  if (n == 0) return DPCLIP_OK;
  DPCLIP_CUDA(launch_philox_fill(out, 1, n, 1, dtype == DPCLIP_BF16, seed, stream_id, offset,
                                 (cudaStream_t)stream));
  return DPCLIP_OK;
}

int dpclip_philox_rademacher(void* out, int64_t n, int dtype, uint64_t seed, uint32_t stream_id,
                             uint64_t offset, dpclip_stream_t stream) {
  if (!out || n < 0) return DPCLIP_ERR_INVALID_ARG;
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  if (!aligned(out, 4)) return DPCLIP_ERR_UNSUPPORTED;
  if (n > (int64_t)4 * 0xFFFFFFFFll) return DPCLIP_ERR_UNSUPPORTED;
  if (n == 0) return DPCLIP_OK;
  DPCLIP_CUDA(launch_philox_fill(out, 1, n, 1, dtype == DPCLIP_BF16, seed, stream_id, offset,
                                 (cudaStream_t)stream, nullptr, 0, DPCLIP_PROBE_RADEMACHER));
  return DPCLIP_OK;
}

int dpclip_clip_scales(const float* sqnorms, int B, float C, float* scales, uint8_t* clipped,
                       dpclip_stream_t stream) {
  if (!sqnorms || B <= 0) return DPCLIP_ERR_INVALID_ARG;
  if (!(C > 0.f) || !std::isfinite(C)) return DPCLIP_ERR_INVALID_ARG;
  if (!scales && !clipped) return DPCLIP_OK;
  DPCLIP_CUDA(launch_clip_scales(sqnorms, B, C, scales, clipped, (cudaStream_t)stream));
  return DPCLIP_OK;
}

int dpclip_norms_exact(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                       int method, float* sqnorms, void* ws, size_t ws_bytes,
                       dpclip_stream_t stream) {
  DPCLIP_TRY(check_shapes(A, G, B, T, d, p, dtype));
  if (!sqnorms) return DPCLIP_ERR_INVALID_ARG;
  Plan pl;
  DPCLIP_TRY(plan_for(DPCLIP_OP_NORMS_EXACT, B, T, d, p, dtype, method, pl));
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  const int m = resolve_exact(method, T, d, p);
  cudaStream_t s = (cudaStream_t)stream;
  DPCLIP_CUDA(launch_clear_words(at<uint32_t>(ws, pl.ctrl), (int)(pl.ctrl_bytes / 4), s));
  if (dtype == DPCLIP_BF16) {
    if (m == DPCLIP_EXACT_DIRECT) {
      GemmDpParams gp;
      std::memset(&gp, 0, sizeof(gp));
      if (!make_map(&gp.map_a, A, d, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
      if (!make_map(&gp.map_g, G, p, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
      gp.B = B;
      gp.T = T;
      gp.d = d;
      gp.p = p;
      gp.mtiles = dp_mtiles(d);
      gp.ntiles = cdiv(p, kDpTileN);
      gp.tblocks = cdiv(T, kBlockK);
      gp.part = at<float>(ws, pl.off[0]);
      gp.sq = sqnorms;
      gp.ticket = at<uint32_t>(ws, pl.ctrl + 4);
      gp.err = at<uint32_t>(ws, pl.ctrl);
      DPCLIP_CUDA(launch_gemm_dp(gp, false, s));
    } else {
      GhostParams gh;
      std::memset(&gh, 0, sizeof(gh));
      if (!make_map(&gh.map_a, A, d, T, B, kBlockK, kGhostTile)) return DPCLIP_ERR_UNSUPPORTED;
      if (!make_map(&gh.map_g, G, p, T, B, kBlockK, kGhostTile)) return DPCLIP_ERR_UNSUPPORTED;
      gh.B = B;
      gh.T = T;
      gh.d = d;
      gh.p = p;
      gh.npairs = ghost_npairs(T);
      gh.dblocks = cdiv(d, kBlockK);
      gh.pblocks = cdiv(p, kBlockK);
      gh.part = at<float>(ws, pl.off[0]);
      gh.xbuf = at<float>(ws, pl.off[1]);
      gh.xready = at<uint32_t>(ws, pl.ctrl + 8);
      gh.sq = sqnorms;
      gh.ticket = at<uint32_t>(ws, pl.ctrl + 4);
      gh.err = at<uint32_t>(ws, pl.ctrl);
      DPCLIP_CUDA(launch_ghost(gh, s));
    }
    return DPCLIP_OK;
  }
  // fp32
  const float* Af = static_cast<const float*>(A);
  const float* Gf = static_cast<const float*>(G);
  SimtParams sp = simt_base();
  int nb = 0;
  if (m == DPCLIP_EXACT_DIRECT) {
    sp.X = Af; sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;     // A_i^T : (f, t)
    sp.Y = Gf; sp.yb = (long long)T * p; sp.yk = p; sp.yn = 1;     // G_i   : (t, c)
    sp.batch = B; sp.M = d; sp.N = p; sp.K = T;
    sp.part = at<float>(ws, pl.off[kFPart]);
    DPCLIP_CUDA(launch_simt(sp, kSimtSqNorm, s, &nb));
  } else {
    float* W = at<float>(ws, pl.off[kFW]);
    sp.X = Af; sp.xb = (long long)T * d; sp.xm = d; sp.xk = 1;     // A_i   : (t, f)
    sp.Y = Af; sp.yb = (long long)T * d; sp.yk = 1; sp.yn = d;     // A_i^T : (f, t2)
    sp.batch = B; sp.M = T; sp.N = T; sp.K = d;
    sp.out = W; sp.ob = (long long)T * T; sp.om = T; sp.on = 1;
    DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
    sp.X = Gf; sp.xb = (long long)T * p; sp.xm = p; sp.xk = 1;
    sp.Y = Gf; sp.yb = (long long)T * p; sp.yk = 1; sp.yn = p;
    sp.K = p;
    sp.part = at<float>(ws, pl.off[kFPart]);
    DPCLIP_CUDA(launch_simt(sp, kSimtDotWith, s, &nb));
  }
  DPCLIP_CUDA(launch_finalize_norms(sp.part, B, nb, 1, nb, 1, 1.f, sqnorms, s));
  return DPCLIP_OK;
}

int dpclip_norms_hutch_ex(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                          int k, int probe, uint64_t seed, uint64_t offset, float* sqnorms,
                          void* ws, size_t ws_bytes, dpclip_stream_t stream) {
  if (probe != DPCLIP_PROBE_GAUSSIAN && probe != DPCLIP_PROBE_RADEMACHER)
    return DPCLIP_ERR_INVALID_ARG;
  DPCLIP_TRY(check_shapes(A, G, B, T, d, p, dtype));
  if (!sqnorms) return DPCLIP_ERR_INVALID_ARG;
  Plan pl;
  DPCLIP_TRY(plan_for(DPCLIP_OP_NORMS_HUTCH, B, T, d, p, dtype, k, pl));
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  cudaStream_t s = (cudaStream_t)stream;
  // the first kernel clears the control block (error word, tickets)
  uint32_t* ctrl = at<uint32_t>(ws, pl.ctrl);
  const int ctrl_words = (int)(pl.ctrl_bytes / 4);
  if (dtype == DPCLIP_BF16) {
    const int NP = np_for(k);
    void* P = at<void>(ws, pl.off[kP]);
    DPCLIP_CUDA(launch_philox_fill(P, NP, p, k, true, seed, 0u, offset, s, ctrl, ctrl_words, probe));
    void* Yhi = at<void>(ws, pl.off[kYhi]);
    void* Ylo = at<void>(ws, pl.off[kYlo]);
    DPCLIP_TRY(run_tok(G, B, T, p, P, nullptr, NP, false, pl, ws, Yhi, Ylo, s));
    float w[kMaxNP];
    for (int j = 0; j < kMaxNP; ++j) w[j] = j < k ? 1.f / (float)k : 0.f;
    DPCLIP_TRY(run_feat(A, B, T, d, Yhi, Ylo, NP, kFeatSqNorm, w, pl, ws,
                        pl.off[kQpart], nullptr, nullptr, nullptr, sqnorms, s));
    return DPCLIP_OK;
  }
  const float* Af = static_cast<const float*>(A);
  const float* Gf = static_cast<const float*>(G);
  float* P = at<float>(ws, pl.off[kFP]);
  float* Y = at<float>(ws, pl.off[kFY]);
  DPCLIP_CUDA(launch_philox_fill(P, k, p, k, false, seed, 0u, offset, s, ctrl, ctrl_words, probe));
  SimtParams sp = simt_base();
  int nb = 0;
  sp.X = Gf; sp.xb = (long long)T * p; sp.xm = p; sp.xk = 1;        // G_i : (t, c)
  sp.Y = P; sp.yb = 0; sp.yk = 1; sp.yn = p;                         // P   : (c, j)
  sp.batch = B; sp.M = T; sp.N = k; sp.K = p;
  sp.out = Y; sp.ob = (long long)T * k; sp.om = k; sp.on = 1;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  sp = simt_base();
  sp.X = Af; sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;         // A_i^T : (f, t)
  sp.Y = Y; sp.yb = (long long)T * k; sp.yk = k; sp.yn = 1;          // Y_i   : (t, j)
  sp.batch = B; sp.M = d; sp.N = k; sp.K = T;
  sp.part = at<float>(ws, pl.off[kFPart]);
  DPCLIP_CUDA(launch_simt(sp, kSimtSqNorm, s, &nb));
  DPCLIP_CUDA(launch_finalize_norms(sp.part, B, nb, 1, nb, 1, 1.f / (float)k, sqnorms, s));
  return DPCLIP_OK;
}

int dpclip_norms_hutchpp_ex(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                            int k, int probe, uint64_t seed, uint64_t offset, float* sqnorms,
                            void* ws, size_t ws_bytes, dpclip_stream_t stream) {
  if (probe != DPCLIP_PROBE_GAUSSIAN && probe != DPCLIP_PROBE_RADEMACHER)
    return DPCLIP_ERR_INVALID_ARG;
  DPCLIP_TRY(check_shapes(A, G, B, T, d, p, dtype));
  if (!sqnorms) return DPCLIP_ERR_INVALID_ARG;
  Plan pl;
  DPCLIP_TRY(plan_for(DPCLIP_OP_NORMS_HUTCHPP, B, T, d, p, dtype, k, pl));
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  const int r = k / 3, m = k - 2 * r;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* ctrl = at<uint32_t>(ws, pl.ctrl);
  const int ctrl_words = (int)(pl.ctrl_bytes / 4);
  float w[kMaxNP];
  for (int j = 0; j < kMaxNP; ++j) w[j] = j < r ? 1.f : (j < r + m ? 1.f / (float)m : 0.f);
  if (dtype == DPCLIP_BF16) {
    void* S = at<void>(ws, pl.off[kS]);
    void* Gp = at<void>(ws, pl.off[kGp]);
    DPCLIP_CUDA(launch_philox_fill2(S, 16, r, 1u, Gp, m, m, 2u, p, true, seed, offset, s, ctrl,
                                    ctrl_words, probe));
    void *Y1h = at<void>(ws, pl.off[kY1hi]), *Y1l = at<void>(ws, pl.off[kY1lo]);
    void *Z1h = at<void>(ws, pl.off[kZ1hi]), *Z1l = at<void>(ws, pl.off[kZ1lo]);
    void *Uh = at<void>(ws, pl.off[kUhi]), *Ul = at<void>(ws, pl.off[kUlo]);
    float* V = at<float>(ws, pl.off[kV]);
    void *QWh = at<void>(ws, pl.off[kQWhi]), *QWl = at<void>(ws, pl.off[kQWlo]);
    void *Y3h = at<void>(ws, pl.off[kY3hi]), *Y3l = at<void>(ws, pl.off[kY3lo]);
    const size_t qpart = pl.off[kHQpart];
    // sweep 1: Y1 = G S, Z1 = A^T Y1
    // G is read once per sweep and A in each of the three: G's loads evict
    // first, so that A (smaller than L2) can stay there between its passes
    DPCLIP_TRY(run_tok(G, B, T, p, S, nullptr, 16, false, pl, ws, Y1h, Y1l, s, true));
    DPCLIP_TRY(run_feat(A, B, T, d, Y1h, Y1l, 16, kFeatOutHiLo, nullptr, pl, ws, qpart,
                        nullptr, Z1h, Z1l, nullptr, s));
    // sweep 2: U = A Z1, V = G^T U  (= O S)
    DPCLIP_TRY(run_tok(A, B, T, d, Z1h, Z1l, 16, true, pl, ws, Uh, Ul, s));
    DPCLIP_TRY(run_feat(G, B, T, p, Uh, Ul, 16, kFeatOutF32, nullptr, pl, ws, qpart, V,
                        nullptr, nullptr, nullptr, s, true, hpp_keep_t0(B, T, d, p)));
    // Q, W
    HppQrParams hq;
    std::memset(&hq, 0, sizeof(hq));
    hq.V = V;
    hq.ldv = 16;
    hq.Gp = Gp;
    hq.gp_bf16 = 1;
    hq.B = B;
    hq.p = p;
    hq.r = r;
    hq.m = m;
    hq.out_hi = static_cast<__nv_bfloat16*>(QWh);
    hq.out_lo = static_cast<__nv_bfloat16*>(QWl);
    hq.err = at<uint32_t>(ws, pl.ctrl);
    DPCLIP_CUDA(launch_hpp_qr(hq, s));
    // sweep 3: Y3 = G [Q | W], head + tail / m from A^T Y3
    DPCLIP_TRY(run_tok(G, B, T, p, QWh, QWl, 32, true, pl, ws, Y3h, Y3l, s, true));
    DPCLIP_TRY(run_feat(A, B, T, d, Y3h, Y3l, 32, kFeatSqNorm, w, pl, ws, qpart, nullptr,
                        nullptr, nullptr, sqnorms, s));
    return DPCLIP_OK;
  }
  const float* Af = static_cast<const float*>(A);
  const float* Gf = static_cast<const float*>(G);
  float* S = at<float>(ws, pl.off[kFS]);
  float* Gp = at<float>(ws, pl.off[kFGp]);
  float* Y1 = at<float>(ws, pl.off[kFY1]);
  float* Z1 = at<float>(ws, pl.off[kFZ1]);
  float* U = at<float>(ws, pl.off[kFU]);
  float* V = at<float>(ws, pl.off[kFV]);
  float* QW = at<float>(ws, pl.off[kFQW]);
  float* Y3 = at<float>(ws, pl.off[kFY3]);
  DPCLIP_CUDA(launch_philox_fill2(S, r, r, 1u, Gp, m, m, 2u, p, false, seed, offset, s, ctrl,
                                  ctrl_words, probe));
  int nb = 0;
  SimtParams sp = simt_base();
  // Y1 = G S
  sp.X = Gf; sp.xb = (long long)T * p; sp.xm = p; sp.xk = 1;
  sp.Y = S; sp.yb = 0; sp.yk = 1; sp.yn = p;
  sp.batch = B; sp.M = T; sp.N = r; sp.K = p;
  sp.out = Y1; sp.ob = (long long)T * r; sp.om = r; sp.on = 1;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  // Z1 = A^T Y1  (d x r)
  sp = simt_base();
  sp.X = Af; sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;
  sp.Y = Y1; sp.yb = (long long)T * r; sp.yk = r; sp.yn = 1;
  sp.batch = B; sp.M = d; sp.N = r; sp.K = T;
  sp.out = Z1; sp.ob = (long long)d * r; sp.om = r; sp.on = 1;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  // U = A Z1  (T x r)
  sp = simt_base();
  sp.X = Af; sp.xb = (long long)T * d; sp.xm = d; sp.xk = 1;
  sp.Y = Z1; sp.yb = (long long)d * r; sp.yk = r; sp.yn = 1;
  sp.batch = B; sp.M = T; sp.N = r; sp.K = d;
  sp.out = U; sp.ob = (long long)T * r; sp.om = r; sp.on = 1;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  // V = G^T U  (p x r), stored [B][16][p]
  sp = simt_base();
  sp.X = Gf; sp.xb = (long long)T * p; sp.xm = 1; sp.xk = p;
  sp.Y = U; sp.yb = (long long)T * r; sp.yk = r; sp.yn = 1;
  sp.batch = B; sp.M = p; sp.N = r; sp.K = T;
  sp.out = V; sp.ob = (long long)16 * p; sp.om = 1; sp.on = p;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  HppQrParams hq;
  std::memset(&hq, 0, sizeof(hq));
  hq.V = V;
  hq.ldv = 16;
  hq.Gp = Gp;
  hq.gp_bf16 = 0;
  hq.B = B;
  hq.p = p;
  hq.r = r;
  hq.m = m;
  hq.out_f32 = QW;
  hq.err = at<uint32_t>(ws, pl.ctrl);
  hq.gram_f64 = 1;
  DPCLIP_CUDA(launch_hpp_qr(hq, s));
  // Y3 = G [Q | W]  (T x (r+m))
  sp = simt_base();
  sp.X = Gf; sp.xb = (long long)T * p; sp.xm = p; sp.xk = 1;
  sp.Y = QW; sp.yb = (long long)32 * p; sp.yk = 1; sp.yn = p;
  sp.batch = B; sp.M = T; sp.N = r + m; sp.K = p;
  sp.out = Y3; sp.ob = (long long)T * (r + m); sp.om = r + m; sp.on = 1;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  // head + tail / m
  sp = simt_base();
  for (int j = 0; j < 64; ++j) sp.w[j] = j < r ? 1.f : (j < r + m ? 1.f / (float)m : 0.f);
  sp.X = Af; sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;
  sp.Y = Y3; sp.yb = (long long)T * (r + m); sp.yk = r + m; sp.yn = 1;
  sp.batch = B; sp.M = d; sp.N = r + m; sp.K = T;
  sp.part = at<float>(ws, pl.off[kFPart]);
  DPCLIP_CUDA(launch_simt(sp, kSimtSqNorm, s, &nb));
  DPCLIP_CUDA(launch_finalize_norms(sp.part, B, nb, 1, nb, 1, 1.f, sqnorms, s));
  return DPCLIP_OK;
}

int dpclip_norms_hutch(const void* A, const void* G, int B, int T, int d, int p, int dtype, int k,
                       uint64_t seed, uint64_t offset, float* sqnorms, void* ws, size_t ws_bytes,
                       dpclip_stream_t stream) {
  return dpclip_norms_hutch_ex(A, G, B, T, d, p, dtype, k, DPCLIP_PROBE_GAUSSIAN, seed, offset,
                               sqnorms, ws, ws_bytes, stream);
}

int dpclip_norms_hutchpp(const void* A, const void* G, int B, int T, int d, int p, int dtype, int k,
                         uint64_t seed, uint64_t offset, float* sqnorms, void* ws, size_t ws_bytes,
                         dpclip_stream_t stream) {
  return dpclip_norms_hutchpp_ex(A, G, B, T, d, p, dtype, k, DPCLIP_PROBE_GAUSSIAN, seed, offset,
                                 sqnorms, ws, ws_bytes, stream);
}

namespace dpclip {
namespace {
// Checks an optional update; *scale = lr / denom.  Returns a status.
int check_update(const dpclip_sgd_update* u, float* scale) {
  *scale = 0.f;
  if (!u) return DPCLIP_OK;
  if (!u->param || (u->store_grad != 0 && u->store_grad != 1)) return DPCLIP_ERR_INVALID_ARG;
  if (!std::isfinite(u->lr) || !(u->denom > 0.f) || !std::isfinite(u->denom))
    return DPCLIP_ERR_INVALID_ARG;
  *scale = u->lr / u->denom;
  return DPCLIP_OK;
}

// Checks an optional FIBER step and converts it for the device.
int make_fiber(const dpclip_fiber_adamw* o, FiberDev* f, bool vec16) {
  if (!o) return DPCLIP_OK;
  if (!o->param || !o->filt || !o->resid || !o->m || !o->v) return DPCLIP_ERR_INVALID_ARG;
  const float hp[] = {o->lr, o->beta1, o->beta2, o->eps, o->eps_v, o->weight_decay, o->omega,
                      o->noise_var, o->denom};
  for (float x : hp)
    if (!std::isfinite(x)) return DPCLIP_ERR_INVALID_ARG;
  if (!(o->omega > 0.f && o->omega <= 1.f) || o->step < 1 || !(o->denom > 0.f) ||
      !(o->beta1 >= 0.f && o->beta1 < 1.f) || !(o->beta2 >= 0.f && o->beta2 < 1.f) ||
      o->eps < 0.f || o->eps_v < 0.f || o->noise_var < 0.f)
    return DPCLIP_ERR_INVALID_ARG;
  const size_t al = vec16 ? 16 : 4;
  if (!aligned(o->param, al) || !aligned(o->filt, al) || !aligned(o->resid, al) ||
      !aligned(o->m, al) || !aligned(o->v, al))
    return DPCLIP_ERR_UNSUPPORTED;
  f->param = o->param;
  f->filt = o->filt;
  f->resid = o->resid;
  f->m = o->m;
  f->v = o->v;
  f->lr = o->lr;
  f->beta1 = o->beta1;
  f->beta2 = o->beta2;
  f->eps = o->eps;
  f->eps_v = o->eps_v;
  f->wd = o->weight_decay;
  f->omega = o->omega;
  f->calib = (float)((2.0 - o->omega) / (4.0 - 3.0 * o->omega) * o->noise_var);
  f->inv_denom = 1.f / o->denom;
  f->bc1 = (float)(1.0 / (1.0 - std::pow((double)o->beta1, o->step)));
  f->bc2 = (float)(1.0 / (1.0 - std::pow((double)o->beta2, o->step)));
  return DPCLIP_OK;
}

int check_noise_args(float C, float sigma) {
  if (!(C > 0.f) || !std::isfinite(C)) return DPCLIP_ERR_INVALID_ARG;
  if (!(sigma >= 0.f) || !std::isfinite(sigma)) return DPCLIP_ERR_INVALID_ARG;
  return DPCLIP_OK;
}

// The clipped noisy gradient from A and G, with at most one of an SGD update
// and a FIBER step fused; grad may be null when neither stores it.
int grad_impl(const void* A, const void* G, int B, int T, int d, int p, int dtype,
              const float* sqnorms, float C, float sigma, uint64_t seed, uint64_t offset,
              float* grad, float* scales, uint8_t* clipped, const dpclip_sgd_update* update,
              const dpclip_fiber_adamw* fopt, void* ws, size_t ws_bytes, cudaStream_t s) {
  float upd_scale;
  DPCLIP_TRY(check_update(update, &upd_scale));
  FiberDev fd{};
  DPCLIP_TRY(make_fiber(fopt, &fd, dtype == DPCLIP_BF16));
  DPCLIP_TRY(check_noise_args(C, sigma));
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  // The FIBER step runs as its own HBM pass over the gradient on this path
  // (inside the GEMM epilogue its five state streams per element stalled the
  // epilogue: 717 us against 382 + 114 us), so grad must be given.
  const bool store = update ? update->store_grad != 0 : true;
  if ((store || dtype == DPCLIP_F32) && !grad) return DPCLIP_ERR_INVALID_ARG;
  float* param = update ? update->param : nullptr;
  const FiberDev* fp = fopt ? &fd : nullptr;
  if (B == 0) {   // an empty lot: the noise alone
    if (d <= 0 || p <= 0) return DPCLIP_ERR_INVALID_ARG;
    DPCLIP_CUDA(launch_noise_only(store ? grad : nullptr, param, (long long)d * p, sigma * C,
                                  upd_scale, seed, 3u, offset, fp, s));
    return DPCLIP_OK;
  }
  DPCLIP_TRY(check_shapes(A, G, B, T, d, p, dtype));
  if (!sqnorms) return DPCLIP_ERR_INVALID_ARG;
  if (grad && !aligned(grad, dtype == DPCLIP_BF16 ? 16 : 4)) return DPCLIP_ERR_UNSUPPORTED;
  if (param && !aligned(param, dtype == DPCLIP_BF16 ? 16 : 4)) return DPCLIP_ERR_UNSUPPORTED;
  Plan pl = plan_grad(d, p, dtype);
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  DPCLIP_CUDA(launch_clear_words(at<uint32_t>(ws, pl.ctrl), (int)(pl.ctrl_bytes / 4), s));
  if (dtype == DPCLIP_BF16) {
    GemmDpParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (!make_map(&gp.map_a, A, d, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
    if (!make_map(&gp.map_g, G, p, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
    gp.B = B;
    gp.T = T;
    gp.d = d;
    gp.p = p;
    gp.mtiles = dp_mtiles(d);
    gp.ntiles = cdiv(p, kDpTileN);
    gp.tblocks = cdiv(T, kBlockK);
    gp.sqnorms = sqnorms;
    gp.C = C;
    gp.sigma = sigma;
    gp.seed = seed;
    gp.offset = offset;
    gp.grad = store ? grad : nullptr;
    gp.scales = scales;
    gp.clipped = clipped;
    gp.upd_param = param;
    gp.upd_scale = upd_scale;
    gp.err = at<uint32_t>(ws, pl.ctrl);
    gp.tickets = at<uint32_t>(ws, pl.ctrl + 4);
    gp.slots = at<float>(ws, pl.off[0]);
    DPCLIP_CUDA(launch_gemm_dp(gp, true, s));
    if (fopt) DPCLIP_CUDA(launch_fiber(grad, (long long)d * p, fd, s));
    return DPCLIP_OK;
  }
  SimtParams sp = simt_base();
  sp.X = static_cast<const float*>(A); sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;
  sp.Y = static_cast<const float*>(G); sp.yb = (long long)T * p; sp.yk = p; sp.yn = 1;
  sp.batch = B; sp.M = d; sp.N = p; sp.K = T;
  sp.out = grad; sp.om = p; sp.on = 1;
  sp.sqnorms = sqnorms;
  sp.C = C;
  DPCLIP_CUDA(launch_simt(sp, kSimtGrad, s, nullptr));
  if (sigma > 0.f)
    DPCLIP_CUDA(launch_noise_add(grad, (long long)d * p, sigma * C, seed, offset, s));
  if (scales || clipped) DPCLIP_CUDA(launch_clip_scales(sqnorms, B, C, scales, clipped, s));
  if (param) DPCLIP_CUDA(launch_sgd_update(param, grad, (long long)d * p, upd_scale, s));
  if (fopt) DPCLIP_CUDA(launch_fiber(grad, (long long)d * p, fd, s));
  return DPCLIP_OK;
}

int stored_grad_impl(int B, int d, int p, const float* sqnorms, float C, float sigma,
                     uint64_t seed, uint64_t offset, float* grad, float* scales, uint8_t* clipped,
                     const dpclip_sgd_update* update, const dpclip_fiber_adamw* fopt,
                     const void* ws, size_t ws_bytes, cudaStream_t s) {
  float upd_scale;
  DPCLIP_TRY(check_update(update, &upd_scale));
  FiberDev fd{};
  DPCLIP_TRY(make_fiber(fopt, &fd, true));
  DPCLIP_TRY(check_noise_args(C, sigma));
  if (B < 0 || d <= 0 || p <= 0) return DPCLIP_ERR_INVALID_ARG;
  const bool store = update ? update->store_grad != 0 : (fopt ? grad != nullptr : true);
  if (store && !grad) return DPCLIP_ERR_INVALID_ARG;
  float* g = store ? grad : nullptr;
  float* param = update ? update->param : nullptr;
  const FiberDev* fp = fopt ? &fd : nullptr;
  if ((g && !aligned(g, 16)) || (param && !aligned(param, 16)) || B > kMaxStoredB)
    return DPCLIP_ERR_UNSUPPORTED;
  if (B == 0) {
    DPCLIP_CUDA(launch_noise_only(g, param, (long long)d * p, sigma * C, upd_scale, seed, 3u,
                                  offset, fp, s));
    return DPCLIP_OK;
  }
  if (!sqnorms) return DPCLIP_ERR_INVALID_ARG;
  const long long stride = (long long)stored_stride(d, p);
  DPCLIP_TRY(check_ws(ws, ws_bytes, kAlign + (size_t)B * stride * 4));
  const float* M = reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws) + kAlign);
  DPCLIP_CUDA(launch_stored_grad(M, B, (long long)d * p, stride, sqnorms, C, sigma * C, seed,
                                 offset, g, scales, clipped, param, upd_scale, fp, s));
  return DPCLIP_OK;
}

int bias_clip_impl(const float* bias_grads, int B, int p, const float* sqnorms, float C,
                   float sigma, uint64_t seed, uint64_t offset, float* grad_b,
                   const dpclip_sgd_update* update, const dpclip_fiber_adamw* fopt,
                   cudaStream_t s) {
  float upd_scale;
  DPCLIP_TRY(check_update(update, &upd_scale));
  FiberDev fd{};
  DPCLIP_TRY(make_fiber(fopt, &fd, false));
  DPCLIP_TRY(check_noise_args(C, sigma));
  if (B < 0 || p <= 0) return DPCLIP_ERR_INVALID_ARG;
  const bool store = update ? update->store_grad != 0 : (fopt ? grad_b != nullptr : true);
  if (store && !grad_b) return DPCLIP_ERR_INVALID_ARG;
  float* g = store ? grad_b : nullptr;
  float* param = update ? update->param : nullptr;
  const FiberDev* fp = fopt ? &fd : nullptr;
  if (B > kMaxStoredB) return DPCLIP_ERR_UNSUPPORTED;
  if (B == 0) {
    DPCLIP_CUDA(launch_noise_only(g, param, p, sigma * C, upd_scale, seed, 4u, offset, fp, s));
    return DPCLIP_OK;
  }
  if (!bias_grads || !sqnorms) return DPCLIP_ERR_INVALID_ARG;
  DPCLIP_CUDA(launch_bias_clip(bias_grads, B, p, sqnorms, C, sigma * C, seed, offset, g, param,
                               upd_scale, fp, s));
  return DPCLIP_OK;
}
}  // namespace
}  // namespace dpclip

int dpclip_clipped_noisy_grad_ex(const void* A, const void* G, int B, int T, int d, int p,
                                 int dtype, const float* sqnorms, float C, float sigma,
                                 uint64_t seed, uint64_t offset, float* grad, float* scales,
                                 uint8_t* clipped, const dpclip_sgd_update* update, void* ws,
                                 size_t ws_bytes, dpclip_stream_t stream) {
  return grad_impl(A, G, B, T, d, p, dtype, sqnorms, C, sigma, seed, offset, grad, scales,
                   clipped, update, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

int dpclip_clipped_noisy_grad_fiber(const void* A, const void* G, int B, int T, int d, int p,
                                    int dtype, const float* sqnorms, float C, float sigma,
                                    uint64_t seed, uint64_t offset, float* grad, float* scales,
                                    uint8_t* clipped, const dpclip_fiber_adamw* opt, void* ws,
                                    size_t ws_bytes, dpclip_stream_t stream) {
  if (!opt) return DPCLIP_ERR_INVALID_ARG;
  return grad_impl(A, G, B, T, d, p, dtype, sqnorms, C, sigma, seed, offset, grad, scales,
                   clipped, nullptr, opt, ws, ws_bytes, (cudaStream_t)stream);
}

int dpclip_clipped_noisy_grad(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                              const float* sqnorms, float C, float sigma, uint64_t seed,
                              uint64_t offset, float* grad, float* scales, uint8_t* clipped,
                              void* ws, size_t ws_bytes, dpclip_stream_t stream) {
  return dpclip_clipped_noisy_grad_ex(A, G, B, T, d, p, dtype, sqnorms, C, sigma, seed, offset,
                                      grad, scales, clipped, nullptr, ws, ws_bytes, stream);
}

int dpclip_norms_direct_store(const void* A, const void* G, int B, int T, int d, int p, int dtype,
                              int accumulate, float* sqnorms, void* ws, size_t ws_bytes,
                              dpclip_stream_t stream) {
  DPCLIP_TRY(check_shapes(A, G, B, T, d, p, dtype));
  if (!sqnorms || (accumulate != 0 && accumulate != 1)) return DPCLIP_ERR_INVALID_ARG;
  const Plan pl = plan_stored(B, d, p, dtype);
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  cudaStream_t s = (cudaStream_t)stream;
  float* M = at<float>(ws, pl.off[0]);
  const long long stride = (long long)stored_stride(d, p);
  DPCLIP_CUDA(launch_clear_words(at<uint32_t>(ws, pl.ctrl), (int)(pl.ctrl_bytes / 4), s));
  if (dtype == DPCLIP_BF16) {
    GemmDpParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (!make_map(&gp.map_a, A, d, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
    if (!make_map(&gp.map_g, G, p, T, B, kBlockK, kBlockK)) return DPCLIP_ERR_UNSUPPORTED;
    gp.B = B;
    gp.T = T;
    gp.d = d;
    gp.p = p;
    gp.mtiles = dp_mtiles(d);
    gp.ntiles = cdiv(p, kDpTileN);
    gp.tblocks = cdiv(T, kBlockK);
    gp.part = at<float>(ws, pl.off[1]);
    gp.sq = sqnorms;
    gp.ticket = at<uint32_t>(ws, pl.ctrl + 4);
    gp.err = at<uint32_t>(ws, pl.ctrl);
    gp.pstore = M;
    gp.accumulate = accumulate;
    DPCLIP_CUDA(launch_gemm_dp(gp, false, s));
    return DPCLIP_OK;
  }
  SimtParams sp = simt_base();
  sp.X = static_cast<const float*>(A); sp.xb = (long long)T * d; sp.xm = 1; sp.xk = d;   // A_i^T
  sp.Y = static_cast<const float*>(G); sp.yb = (long long)T * p; sp.yk = p; sp.yn = 1;   // G_i
  sp.batch = B; sp.M = d; sp.N = p; sp.K = T;
  sp.out = M; sp.ob = stride; sp.om = p; sp.on = 1;
  int nb = 0;
  DPCLIP_CUDA(launch_simt(sp, kSimtStore, s, &nb));
  float* part = at<float>(ws, pl.off[1]);
  DPCLIP_CUDA(launch_stored_sqnorm(M, B, (long long)d * p, stride, kStoredSqBlocks, part, s));
  DPCLIP_CUDA(launch_finalize_norms(part, B, kStoredSqBlocks, 1, kStoredSqBlocks, 1, 1.f, sqnorms,
                                    s, accumulate));
  return DPCLIP_OK;
}

int dpclip_stored_clipped_noisy_grad_ex(int B, int d, int p, const float* sqnorms, float C,
                                        float sigma, uint64_t seed, uint64_t offset, float* grad,
                                        float* scales, uint8_t* clipped,
                                        const dpclip_sgd_update* update, const void* ws,
                                        size_t ws_bytes, dpclip_stream_t stream) {
  return stored_grad_impl(B, d, p, sqnorms, C, sigma, seed, offset, grad, scales, clipped, update,
                          nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

int dpclip_stored_clipped_noisy_grad_fiber(int B, int d, int p, const float* sqnorms, float C,
                                           float sigma, uint64_t seed, uint64_t offset,
                                           float* grad, float* scales, uint8_t* clipped,
                                           const dpclip_fiber_adamw* opt, const void* ws,
                                           size_t ws_bytes, dpclip_stream_t stream) {
  if (!opt) return DPCLIP_ERR_INVALID_ARG;
  return stored_grad_impl(B, d, p, sqnorms, C, sigma, seed, offset, grad, scales, clipped, nullptr,
                          opt, ws, ws_bytes, (cudaStream_t)stream);
}

int dpclip_stored_clipped_noisy_grad(int B, int d, int p, const float* sqnorms, float C,
                                     float sigma, uint64_t seed, uint64_t offset, float* grad,
                                     float* scales, uint8_t* clipped, const void* ws,
                                     size_t ws_bytes, dpclip_stream_t stream) {
  if (B <= 0) return DPCLIP_ERR_INVALID_ARG;
  return dpclip_stored_clipped_noisy_grad_ex(B, d, p, sqnorms, C, sigma, seed, offset, grad,
                                             scales, clipped, nullptr, ws, ws_bytes, stream);
}

int dpclip_bias_grads(const void* G, int B, int T, int p, int dtype, int accumulate,
                      float* sqnorms, float* bias_grads, void* ws, size_t ws_bytes,
                      dpclip_stream_t stream) {
  if (!G || B <= 0 || T <= 0 || p <= 0) return DPCLIP_ERR_INVALID_ARG;
  if (dtype != DPCLIP_F32 && dtype != DPCLIP_BF16) return DPCLIP_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return DPCLIP_ERR_INVALID_ARG;
  if (!sqnorms && !bias_grads) return DPCLIP_ERR_INVALID_ARG;
  if (dtype == DPCLIP_BF16 && (p % 8 != 0 || !aligned(G, 16))) return DPCLIP_ERR_UNSUPPORTED;
  if (dtype == DPCLIP_F32 && !aligned(G, 4)) return DPCLIP_ERR_UNSUPPORTED;
  Plan pl;
  DPCLIP_TRY(plan_for(DPCLIP_OP_BIAS, B, T, 1, p, dtype, 0, pl));
  DPCLIP_TRY(check_ws(ws, ws_bytes, pl.total));
  DPCLIP_CUDA(launch_bias_grads(G, dtype == DPCLIP_BF16, B, T, p, at<float>(ws, pl.off[0]),
                                bias_grads, sqnorms, accumulate, (cudaStream_t)stream));
  return DPCLIP_OK;
}

int dpclip_clipped_noisy_bias_grad_ex(const float* bias_grads, int B, int p, const float* sqnorms,
                                      float C, float sigma, uint64_t seed, uint64_t offset,
                                      float* grad_b, const dpclip_sgd_update* update,
                                      dpclip_stream_t stream) {
  return bias_clip_impl(bias_grads, B, p, sqnorms, C, sigma, seed, offset, grad_b, update, nullptr,
                        (cudaStream_t)stream);
}

int dpclip_clipped_noisy_bias_grad_fiber(const float* bias_grads, int B, int p,
                                         const float* sqnorms, float C, float sigma,
                                         uint64_t seed, uint64_t offset, float* grad_b,
                                         const dpclip_fiber_adamw* opt, dpclip_stream_t stream) {
  if (!opt) return DPCLIP_ERR_INVALID_ARG;
  return bias_clip_impl(bias_grads, B, p, sqnorms, C, sigma, seed, offset, grad_b, nullptr, opt,
                        (cudaStream_t)stream);
}

int dpclip_clipped_noisy_bias_grad(const float* bias_grads, int B, int p, const float* sqnorms,
                                   float C, float sigma, uint64_t seed, uint64_t offset,
                                   float* grad_b, dpclip_stream_t stream) {
  if (B <= 0) return DPCLIP_ERR_INVALID_ARG;
  return dpclip_clipped_noisy_bias_grad_ex(bias_grads, B, p, sqnorms, C, sigma, seed, offset,
                                           grad_b, nullptr, stream);
}

int dpclip_fiber_adamw_step(const float* grad, int64_t n, const dpclip_fiber_adamw* opt,
                            dpclip_stream_t stream) {
  if (!grad || n <= 0 || !opt) return DPCLIP_ERR_INVALID_ARG;
  FiberDev fd{};
  DPCLIP_TRY(make_fiber(opt, &fd, false));
  if (!aligned(grad, 4)) return DPCLIP_ERR_UNSUPPORTED;
  DPCLIP_CUDA(launch_fiber(grad, n, fd, (cudaStream_t)stream));
  return DPCLIP_OK;
}

int dpclip_workspace_status(const void* ws, dpclip_stream_t stream) {
  if (!ws) return DPCLIP_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return DPCLIP_ERR_CUDA;
  }
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    (void)cudaGetLastError();
    return DPCLIP_ERR_CUDA;
  }
  return (int)word;
}

int dpclip_grad_tail_schedule(int pairs, int ntiles, int B, int tblocks, int* waves, int* ntail,
                              int64_t* segs, int seg_cap, int* nsegs, int64_t* contrib,
                              int contrib_cap, int* ncontrib) {
  if (pairs < 1 || pairs > kMaxPersistentGrid / 2 || ntiles < 1 || B < 1 || tblocks < 1 ||
      !waves || !ntail || !nsegs || !ncontrib || seg_cap < 0 || contrib_cap < 0 ||
      (seg_cap > 0 && !segs) || (contrib_cap > 0 && !contrib))
    return DPCLIP_ERR_INVALID_ARG;
  uint32_t cover = 0;
  plan_grad_schedule(ntiles, B, tblocks, pairs, *waves, *ntail, cover);
  grad_tail_dump(pairs, *ntail, (long long)B * tblocks, cover, segs, seg_cap, nsegs, contrib,
                 contrib_cap, ncontrib);
  return DPCLIP_OK;
}

int dpclip_ghost_schedule(int pairs, int B, int T, int d, int p, int* nfull, int* tail_split,
                          int* pb_per_split, int* tail_shared) {
  if (pairs < 1 || pairs > kMaxPersistentGrid / 2 || B < 1 || T < 1 || d < 1 || p < 1 || !nfull ||
      !tail_split || !pb_per_split || !tail_shared)
    return DPCLIP_ERR_INVALID_ARG;
  GhostParams gh;
  std::memset(&gh, 0, sizeof(gh));
  gh.B = B;
  gh.npairs = ghost_npairs(T);
  gh.dblocks = cdiv(d, kBlockK);
  gh.pblocks = cdiv(p, kBlockK);
  plan_ghost_schedule(gh, std::min(pairs, B * gh.npairs));
  *nfull = gh.nfull;
  *tail_split = gh.tail_split;
  *pb_per_split = gh.pb_per_split;
  *tail_shared = gh.tail_shared;
  return DPCLIP_OK;
}

int dpclip_selftest_wait_timeout(void* ws, size_t ws_bytes, int timeout_us, dpclip_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return DPCLIP_ERR_INVALID_ARG;
  DPCLIP_TRY(check_ws(ws, ws_bytes, kAlign));
  cudaStream_t s = (cudaStream_t)stream;
  DPCLIP_CUDA(cudaMemsetAsync(ws, 0, kAlign, s));
  DPCLIP_CUDA(launch_wait_selftest(static_cast<uint32_t*>(ws), (uint64_t)timeout_us * 1000ull, s));
  return DPCLIP_OK;
}

}  // extern "C"
