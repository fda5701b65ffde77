// pb_api.cu — the C ABI (include/pb.h): argument checks, workspace and scratch layout,
// TMA tensor maps, and the launch sequence of one parallel block
//   LN -> GEMM [Wqkv | W1] (+GeLU) -> sliding-window attention -> GEMM [Wo ; W2] (+x)
// (MegaScale reading notes, section 1.1, eq. (4)). All device memory belongs to the
// caller; this file allocates none.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/pb.h"
#include "kernels.h"

using pb::EpiParams;

struct pb_handle {
  uint32_t magic;
  pb_dims d;
  int device;
  int num_sms;
  uint64_t limit_ns;
  uint8_t* ws;
  int* status;             // device status word
  bool f16;                // PB_OPERANDS_FP16: 16-bit intermediates and weights are fp16
  bool fp8;                // PB_OPERANDS_FP8: the GEMMs take E4M3 operands
  pb::OpType op16;         // type of the 16-bit intermediates (bf16 or fp16)
  pb::OpType gop;          // operand type of the GEMMs
  void* w1cat;             // [3H + F, H], bf16, fp16 or E4M3 codes
  void* w2cat;             // [H, H + F], bf16, fp16 or E4M3 codes
  float* w1scale;          // FP8: [3H + F] per-output-channel scales of W1cat
  float* w2scale;          // FP8: [H] per-output-channel scales of W2cat
  float* bias1;            // [3H + F]
  float* bias2;            // [H] = b_o + b2
  float* bias_o;           // [H] = b_o (serial block)
  float* bias_2;           // [H] = b2 (serial block)
  __nv_bfloat16* gamma;    // [H]
  __nv_bfloat16* beta;     // [H]
  bool has_bias;
  CUtensorMap tm_w1cat;
  CUtensorMap tm_w2cat;
  std::vector<cudaEvent_t> trace;  // 5 events per traced call
  int trace_max;
  int trace_calls;
  // pb_forward_stack_host_steps (created on first use, in the stack's first handle): the
  // copy stream and its events (start, input ready x2, compute done x2, output done)
  cudaStream_t copy_stream;
  cudaEvent_t copy_ev[6];
};

namespace {

constexpr uint32_t kMagic = 0x50424C4Bu;  // "PBLK"
constexpr uint32_t kDead = 0xDEADB10Cu;
constexpr uint64_t kDefaultLimitNs = 2000000000ull;

thread_local std::string g_last_error;

pb_status fail(pb_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

pb_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define PB_CUDA(call, what)                      \
  do {                                           \
    cudaError_t e_ = (call);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bytes left unused after every region of the weight workspace and of the scratch layouts
// (pb_set_guard_bytes; 0 by default). A test fills them with a canary and checks them after
// its calls: a kernel that writes past the end of a region changes them.
std::atomic<size_t> g_guard_bytes{0};

// Next region offset after a region of `bytes` at `off`: the guard gap, then 1024-byte
// alignment.
size_t next_region(size_t off, size_t bytes) {
  return align_up(off + bytes + g_guard_bytes.load(std::memory_order_relaxed), 1024);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pb_status check_dims(const pb_dims* d) {
  if (d == nullptr) return fail(PB_ERR_INVALID_ARG, "dims is NULL");
  if (d->batch < 1 || d->seq < 1 || d->hidden < 1 || d->heads < 1 || d->head_dim < 1 ||
      d->ffn < 1 || d->window < 1)
    return fail(PB_ERR_INVALID_ARG, "every dimension must be >= 1");
  if (!(d->ln_eps > 0.f) || !std::isfinite(d->ln_eps))
    return fail(PB_ERR_INVALID_ARG, "ln_eps must be finite and > 0");
  if (int64_t(d->heads) * d->head_dim != d->hidden)
    return fail(PB_ERR_INVALID_ARG, "hidden (%d) != heads (%d) * head_dim (%d)", d->hidden,
                d->heads, d->head_dim);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PB_ERR_UNSUPPORTED, "head_dim %d: supported are 64 and 128", d->head_dim);
  if (d->hidden % 64 != 0 || d->ffn % 64 != 0)
    return fail(PB_ERR_UNSUPPORTED, "hidden and ffn must be multiples of 64");
  if (d->hidden > pb::kLnMaxH)
    return fail(PB_ERR_UNSUPPORTED, "hidden %d > %d", d->hidden, pb::kLnMaxH);
  const int64_t T = int64_t(d->batch) * d->seq;
  if (T >= (int64_t(1) << 31)) return fail(PB_ERR_UNSUPPORTED, "batch * seq >= 2^31");
  if (int64_t(3) * d->hidden + 2 * int64_t(d->ffn) >= (int64_t(1) << 31))
    return fail(PB_ERR_UNSUPPORTED, "3 * hidden + 2 * ffn >= 2^31");
  if (d->variant != PB_BLOCK_LN_GELU && d->variant != PB_BLOCK_RMS_SWIGLU)
    return fail(PB_ERR_INVALID_ARG, "variant %d is not a pb_block_variant", d->variant);
  return PB_OK;
}

bool is_glu(const pb_dims& d) { return d.variant == PB_BLOCK_RMS_SWIGLU; }

// Output columns of the first GEMM / rows of W1cat: [q | k | v | h], h = F columns (GeLU)
// or 2F (SwiGLU gate and up, interleaved).
int64_t w1_rows(const pb_dims& d) {
  return 3 * int64_t(d.hidden) + (is_glu(d) ? 2 : 1) * int64_t(d.ffn);
}

struct WsLayout {
  size_t status, w1cat, w2cat, bias1, bias2, bias_o, bias_2, gamma, beta;
  size_t w1scale, w2scale, amax1, amax2;  // FP8 operands (reserved in every mode)
  size_t total;
};

WsLayout ws_layout(const pb_dims& d) {
  const size_t H = size_t(d.hidden), F = size_t(d.ffn);
  WsLayout L{};
  size_t off = 0;
  L.status = off;
  off = next_region(off, 256);
  L.w1cat = off;
  off = next_region(off, size_t(w1_rows(d)) * H * 2);
  L.w2cat = off;
  off = next_region(off, H * (H + F) * 2);
  L.bias1 = off;
  off = next_region(off, size_t(w1_rows(d)) * 4);
  L.bias2 = off;
  off = next_region(off, H * 4);
  L.bias_o = off;
  off = next_region(off, H * 4);
  L.bias_2 = off;
  off = next_region(off, H * 4);
  L.gamma = off;
  off = next_region(off, H * 2);
  L.beta = off;
  off = next_region(off, H * 2);
  L.w1scale = off;
  off = next_region(off, size_t(w1_rows(d)) * 4);
  L.w2scale = off;
  off = next_region(off, H * 4);
  L.amax1 = off;
  off = next_region(off, size_t(w1_rows(d)) * 4);
  L.amax2 = off;
  off = next_region(off, H * 4);
  L.total = off;
  return L;
}

// Row stride of the per-row attention values of training (log-sum-exp, D): the sequence
// rounded up to 64, so the backward's 64-row copies of them stay inside a row.
size_t lse_ld(const pb_dims& d) { return align_up(size_t(d.seq), 64); }

pb_scratch_layout scratch_layout(const pb_dims& d) {
  const size_t H = size_t(d.hidden), F = size_t(d.ffn);
  const size_t T = size_t(d.batch) * size_t(d.seq);
  pb_scratch_layout L{};
  L.seq_pad = align_up(size_t(d.seq), 8);
  size_t off = 0;
  L.xn = off;
  off = next_region(off, T * H * 2);
  L.qk = off;
  off = next_region(off, T * 2 * H * 2);
  L.vt = off;
  off = next_region(off, size_t(d.batch) * H * L.seq_pad * 2);
  L.act = off;
  off = next_region(off, T * (H + F) * 2);
  L.io = off;
  off = next_region(off, T * H * 2);
  L.io2 = off;
  off = next_region(off, T * H * 2);
  L.res0 = off;
  off = next_region(off, T * H * 4);
  L.res1 = off;
  off = next_region(off, T * H * 4);
  L.sk = off;
  off = next_region(off, pb::kSkScratchBytes);
  L.q8 = off;
  off = next_region(off, T * (H + F));
  L.qscale = off;
  off = next_region(off, 2 * T * 4);
  L.total = off;
  // training: what the backward reads from the forward, then its own intermediates
  const size_t Fp = size_t(w1_rows(d)) - 3 * H;  // F, or 2F for SwiGLU
  const size_t NZ = size_t(w1_rows(d));          // columns of dz = [dq | dk | dv | dh]
  const size_t rows_lse = size_t(d.batch) * size_t(d.heads) * lse_ld(d);
  L.hpre = off;
  off = next_region(off, T * Fp * 2);
  L.lse = off;
  off = next_region(off, rows_lse * 4);
  L.d_attn = off;
  off = next_region(off, T * H * 2);
  L.delta = off;
  off = next_region(off, rows_lse * 4);
  L.dq_acc = off;
  off = next_region(off, T * H * 4);
  L.dz = off;
  off = next_region(off, T * NZ * 2);
  L.dxn = off;
  off = next_region(off, T * H * 4);
  L.stats = off;
  off = next_region(off, T * 8);
  L.partials = off;
  off = next_region(off, size_t(pb::kColBlocks) * (NZ > 2 * H ? NZ : 2 * H) * 4);
  L.train_total = off;
  return L;
}

// ---------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

pb_status get_encoder(EncodeTiledFn* out) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static cudaError_t err = cudaSuccess;
  static cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                           cudaEnableDefault, &q);
    fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDriverEntryPointByVersion");
  if (fn == nullptr || q != cudaDriverEntryPointSuccess)
    return fail(PB_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  *out = fn;
  return PB_OK;
}

CUtensorMapDataType map_type(pb::OpType t) {
  switch (t) {
    case pb::kOpF16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case pb::kOpE4m3: return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // raw E4M3 bytes
    default: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  }
}

// Tensor of `rank` dims (dims[0] innermost) of element type t, 128-byte swizzle, zero fill
// outside.
pb_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box,
                   pb::OpType t = pb::kOpBf16) {
  EncodeTiledFn enc;
  pb_status s = get_encoder(&enc);
  if (s != PB_OK) return s;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = enc(m, map_type(t), cuuint32_t(rank), const_cast<void*>(base),
                   gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PB_OK;
}

// fp32 tensor of `rank` dims, no swizzle (boxes land row-major in shared memory).
pb_status make_map_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn enc;
  pb_status s = get_encoder(&enc);
  if (s != PB_OK) return s;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cuuint32_t(rank), const_cast<void*>(base),
                   gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PB_OK;
}

// Row-major [rows, cols] 16-bit output (bf16, or fp16 when f16) written by the GEMM
// epilogues' TMA stores: boxes of 32 columns x 32 rows with 64-byte swizzle (one epilogue
// warp's chunk).
pb_status make_store_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint64_t ld, bool f16) {
  EncodeTiledFn enc;
  pb_status s = get_encoder(&enc);
  if (s != PB_OK) return s;
  const cuuint64_t gd[2] = {cols, rows};
  const cuuint64_t gs[1] = {ld * 2};
  const cuuint32_t bx[2] = {32, 32}, es[2] = {1, 1};
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PB_OK;
}

// Row-major [rows, cols] matrix of element type t read in boxes of 128 bytes of columns
// (64 16-bit or 128 FP8 elements) x box_rows rows.
pb_status make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint64_t ld, uint32_t box_rows, pb::OpType t = pb::kOpBf16) {
  const uint64_t esz = t == pb::kOpE4m3 ? 1 : 2;
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {ld * esz};
  const uint32_t box[2] = {uint32_t(128 / esz), box_rows};
  return make_map(m, base, 2, dims, strides, box, t);
}

// Tensor maps of the attention step: q|k [B][S][2H] read as query tiles and as key tiles,
// and v^T [B*H][seq_pad] read in boxes of 64 keys x dh rows.
pb_status make_swa_maps(const pb_dims& d, const void* qk, const void* vt, size_t seq_pad,
                        CUtensorMap* tm_q, CUtensorMap* tm_k, CUtensorMap* tm_vt) {
  const uint64_t H = uint64_t(d.hidden);
  const uint64_t dims[3] = {2 * H, uint64_t(d.seq), uint64_t(d.batch)};
  const uint64_t strides[2] = {2 * H * 2, 2 * H * 2 * uint64_t(d.seq)};
  const uint32_t qbox[3] = {64, uint32_t(pb::kSwaBQ), 1};
  const uint32_t kbox[3] = {64, uint32_t(pb::kSwaBKV), 1};
  pb_status s = make_map(tm_q, qk, 3, dims, strides, qbox);
  if (s == PB_OK) s = make_map(tm_k, qk, 3, dims, strides, kbox);
  if (s != PB_OK) return s;
  const uint64_t vdims[2] = {uint64_t(d.seq), uint64_t(d.batch) * H};
  const uint64_t vstr[1] = {uint64_t(seq_pad) * 2};
  const uint32_t vbox[2] = {64, uint32_t(d.head_dim)};  // 64 keys = one 128-byte swizzle row
  return make_map(tm_vt, vt, 2, vdims, vstr, vbox);
}

pb_status check_handle(pb_handle* h) {
  if (h == nullptr) return fail(PB_ERR_BAD_HANDLE, "handle is NULL");
  if (h->magic != kMagic) return fail(PB_ERR_BAD_HANDLE, "handle is destroyed or invalid");
  int dev = -1;
  PB_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != h->device)
    return fail(PB_ERR_BAD_HANDLE, "handle belongs to device %d, current device is %d", h->device,
                dev);
  return PB_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// One block from x to y (each bf16, or fp32 inside a stack's residual stream),
// intermediates in `scratch`.
pb_status run_block(pb_handle* h, const void* x, bool x_f32, void* y, bool y_f32,
                    uint8_t* scratch, cudaStream_t st, bool train = false) {
  const pb_dims& d = h->d;
  const pb_scratch_layout L = scratch_layout(d);
  const int H = d.hidden, F = d.ffn, T = d.batch * d.seq;
  void* xn = scratch + L.xn;
  auto* qk = reinterpret_cast<__nv_bfloat16*>(scratch + L.qk);
  auto* vt = reinterpret_cast<__nv_bfloat16*>(scratch + L.vt);
  void* act = scratch + L.act;

  cudaEvent_t* ev = nullptr;
  if (h->trace_calls < h->trace_max) ev = &h->trace[size_t(h->trace_calls++) * 5];
  auto mark = [&](int i) -> cudaError_t { return ev ? cudaEventRecord(ev[i], st) : cudaSuccess; };
  PB_CUDA(mark(0), "cudaEventRecord");

  // 1. the shared LayerNorm (RMSNorm for the SwiGLU variant: no beta); with FP8 operands
  // it writes E4M3 codes of LN(x) and their per-row scales
  const bool glu = is_glu(d);
  float* qscale = reinterpret_cast<float*>(scratch + L.qscale);
  if (h->fp8)
    PB_CUDA(pb::launch_layernorm_e4m3(T, H, x, x_f32, h->gamma, glu ? nullptr : h->beta,
                                      d.ln_eps, static_cast<uint8_t*>(xn), qscale, st),
            "layernorm launch");
  else
    PB_CUDA(pb::launch_layernorm(T, H, x, x_f32, h->gamma, glu ? nullptr : h->beta, d.ln_eps,
                                 xn, h->f16, h->status, st),
            "layernorm launch");
  PB_CUDA(mark(1), "cudaEventRecord");

  // 2. [q | k | v | h] = xn [Wqkv | W1], GeLU(h) in the epilogue
  CUtensorMap tm_xn, tm_act, tm_qk, tm_vt;
  pb_status s = make_map_2d(&tm_xn, xn, T, H, H, pb::kGemmBoxRows, h->gop);
  if (s != PB_OK) return s;
  EpiParams e1{};
  e1.status = h->status;
  e1.H = H;
  e1.F = F;
  e1.S = d.seq;
  e1.nh = d.heads;
  e1.dh = d.head_dim;
  e1.seq_pad = int64_t(L.seq_pad);
  e1.qk = qk;
  e1.vt = vt;
  e1.act = act;
  e1.act_f16 = h->f16;
  e1.bias = h->has_bias ? h->bias1 : nullptr;
  e1.glu = glu;
  if (h->fp8) {
    e1.scale_a = qscale;
    e1.scale_b = h->w1scale;
  }
  if (train) e1.hpre = reinterpret_cast<__nv_bfloat16*>(scratch + L.hpre);
  if (!glu) {  // q|k and GeLU(h) by TMA stores (SwiGLU's 16-column outputs stay row stores)
    s = make_store_map(&e1.tm_out0, qk, T, 2 * uint64_t(H), 2 * uint64_t(H), false);
    if (s == PB_OK) s = make_store_map(&e1.tm_out1, act, T, uint64_t(H + F), uint64_t(H + F), h->f16);
    if (s != PB_OK) return s;
    e1.tma_store = true;
  }
  PB_CUDA(pb::launch_gemm(pb::kEpiBlockIn, h->gop, tm_xn, h->tm_w1cat, T, int(w1_rows(d)), H,
                          e1, h->num_sms, h->status, h->limit_ns, scratch + L.sk, st),
          "first GEMM launch");
  PB_CUDA(mark(2), "cudaEventRecord");

  // 3. sliding-window attention -> act[:, 0:H]
  CUtensorMap tm_k;
  s = make_swa_maps(d, qk, vt, L.seq_pad, &tm_qk, &tm_k, &tm_vt);
  if (s != PB_OK) return s;
  pb::SwaParams sp{};
  sp.B = d.batch;
  sp.S = d.seq;
  sp.H = H;
  sp.nh = d.heads;
  sp.dh = d.head_dim;
  sp.window = d.window;
  sp.num_q_tiles = (d.seq + pb::kSwaBQ - 1) / pb::kSwaBQ;
  sp.scale_log2 = float(1.4426950408889634 / std::sqrt(double(d.head_dim)));
  sp.out = act;
  sp.out_ld = H + F;
  sp.out_f16 = h->f16;
  if (train) {
    sp.lse = reinterpret_cast<float*>(scratch + L.lse);
    sp.lse_ld = int64_t(lse_ld(d));
  }
  PB_CUDA(pb::launch_swa(tm_qk, tm_k, tm_vt, sp, h->status, h->limit_ns, st), "attention launch");
  PB_CUDA(mark(3), "cudaEventRecord");

  // 4. y = x + [attn | GeLU(h)] [Wo ; W2] (+ b_o + b2). With FP8 operands the rows of
  // act are quantized first (per-row scales in qscale[T, 2T); timed with this step).
  const void* a2 = act;
  if (h->fp8) {
    uint8_t* q8 = scratch + L.q8;
    PB_CUDA(pb::launch_quantize_rows_e4m3(static_cast<const __nv_bfloat16*>(act), T, H + F,
                                          H + F, q8, H + F, qscale + T, st),
            "act quantization launch");
    a2 = q8;
  }
  s = make_map_2d(&tm_act, a2, T, H + F, H + F, pb::kGemmBoxRows, h->gop);
  if (s != PB_OK) return s;
  EpiParams e2{};
  e2.status = h->status;
  e2.bias = h->has_bias ? h->bias2 : nullptr;
  e2.resid = x;
  e2.resid_f32 = x_f32;
  e2.y = y;
  e2.y_f32 = y_f32;
  if (h->fp8) {
    e2.scale_a = qscale + T;
    e2.scale_b = h->w2scale;
  }
  if (!y_f32) {  // bf16 y by TMA stores
    s = make_store_map(&e2.tm_out0, y, T, uint64_t(H), uint64_t(H), false);
    if (s != PB_OK) return s;
    e2.tma_store = true;
  }
  PB_CUDA(pb::launch_gemm(pb::kEpiResidual, h->gop, tm_act, h->tm_w2cat, T, H, H + F, e2,
                          h->num_sms, h->status, h->limit_ns, scratch + L.sk, st),
          "second GEMM launch");
  PB_CUDA(mark(4), "cudaEventRecord");
  return PB_OK;
}

// The serial (standard) block of eq. (3) on the same packed weights, for comparison with
// the parallel block (MegaScale reading notes, section 1.1):
//   h = x + Attn(LN(x))        (fp32, scratch res0)
//   y = h + MLP(LN'(h))
// Seven launches: LN, GEMM over the Wqkv rows of W1cat, attention, GEMM over the Wo
// columns of W2cat (+ x), LN', GEMM over the W1 rows of W1cat (GeLU), GEMM over the W2
// columns of W2cat (+ h). The two output projections cannot share one GEMM here: the MLP
// reads LN'(h), which needs the attention output first.
pb_status run_serial(pb_handle* h, const void* x, void* y, const __nv_bfloat16* gamma2,
                     const __nv_bfloat16* beta2, uint8_t* scratch, cudaStream_t st) {
  const pb_dims& d = h->d;
  const pb_scratch_layout L = scratch_layout(d);
  const int H = d.hidden, F = d.ffn, T = d.batch * d.seq;
  const uint32_t box = pb::kGemmBoxRows;
  const size_t esz = 2;  // bf16 or fp16 operands
  void* xn = scratch + L.xn;
  auto* qk = reinterpret_cast<__nv_bfloat16*>(scratch + L.qk);
  auto* vt = reinterpret_cast<__nv_bfloat16*>(scratch + L.vt);
  uint8_t* act = scratch + L.act;
  float* hres = reinterpret_cast<float*>(scratch + L.res0);
  uint8_t* w1c = static_cast<uint8_t*>(h->w1cat);
  uint8_t* w2c = static_cast<uint8_t*>(h->w2cat);

  // 1. LN(x) (RMSNorm for the SwiGLU variant)
  const bool glu = is_glu(d);
  PB_CUDA(pb::launch_layernorm(T, H, x, false, h->gamma, glu ? nullptr : h->beta, d.ln_eps, xn,
                               h->f16, h->status, st),
          "layernorm launch");
  // 2. [q | k | v] = xn Wqkv (+ b_qkv): rows [0, 3H) of W1cat
  CUtensorMap tm_xn, tm_wqkv;
  pb_status s = make_map_2d(&tm_xn, xn, T, H, H, box, h->op16);
  if (s == PB_OK) s = make_map_2d(&tm_wqkv, w1c, 3 * uint64_t(H), H, H, box, h->op16);
  if (s != PB_OK) return s;
  EpiParams e1{};
  e1.status = h->status;
  e1.H = H;
  e1.F = F;
  e1.S = d.seq;
  e1.nh = d.heads;
  e1.dh = d.head_dim;
  e1.seq_pad = int64_t(L.seq_pad);
  e1.qk = qk;
  e1.vt = vt;
  e1.act = act;
  e1.act_f16 = h->f16;
  e1.bias = h->has_bias ? h->bias1 : nullptr;
  e1.glu = glu;
  PB_CUDA(pb::launch_gemm(pb::kEpiBlockIn, h->op16, tm_xn, tm_wqkv, T, 3 * H, H, e1, h->num_sms,
                          h->status, h->limit_ns, scratch + L.sk, st),
          "QKV GEMM launch");
  // 3. sliding-window attention -> act[:, 0:H]
  CUtensorMap tm_qk, tm_k, tm_vt;
  s = make_swa_maps(d, qk, vt, L.seq_pad, &tm_qk, &tm_k, &tm_vt);
  if (s != PB_OK) return s;
  pb::SwaParams sp{};
  sp.B = d.batch;
  sp.S = d.seq;
  sp.H = H;
  sp.nh = d.heads;
  sp.dh = d.head_dim;
  sp.window = d.window;
  sp.num_q_tiles = (d.seq + pb::kSwaBQ - 1) / pb::kSwaBQ;
  sp.scale_log2 = float(1.4426950408889634 / std::sqrt(double(d.head_dim)));
  sp.out = act;
  sp.out_ld = H + F;
  sp.out_f16 = h->f16;
  PB_CUDA(pb::launch_swa(tm_qk, tm_k, tm_vt, sp, h->status, h->limit_ns, st), "attention launch");
  // 4. h = x + attn Wo (+ b_o): columns [0, H) of W2cat, result in fp32
  CUtensorMap tm_attn, tm_wo;
  s = make_map_2d(&tm_attn, act, T, H, H + F, box, h->op16);
  if (s == PB_OK) s = make_map_2d(&tm_wo, w2c, H, H, H + F, box, h->op16);
  if (s != PB_OK) return s;
  EpiParams e2{};
  e2.status = h->status;
  e2.bias = h->has_bias ? h->bias_o : nullptr;
  e2.resid = x;
  e2.resid_f32 = false;
  e2.y = hres;
  e2.y_f32 = true;
  PB_CUDA(pb::launch_gemm(pb::kEpiResidual, h->op16, tm_attn, tm_wo, T, H, H, e2, h->num_sms,
                          h->status, h->limit_ns, scratch + L.sk, st),
          "attention projection GEMM launch");
  // 5. LN'(h) -> xn
  PB_CUDA(pb::launch_layernorm(T, H, hres, true, gamma2, glu ? nullptr : beta2, d.ln_eps, xn,
                               h->f16, h->status, st),
          "second layernorm launch");
  // 6. GeLU(LN'(h) W1 (+ b1)) (or SwiGLU) -> act[:, H:H+F]: rows [3H, 3H + F) of W1cat
  // ([3H, 3H + 2F) for SwiGLU), routed as the h columns of [q | k | v | h]
  const int n_h = int(w1_rows(d) - 3 * int64_t(H));
  CUtensorMap tm_w1;
  s = make_map_2d(&tm_w1, w1c + 3 * size_t(H) * H * esz, n_h, H, H, box, h->op16);
  if (s != PB_OK) return s;
  EpiParams e3 = e1;
  e3.col_base = 3 * H;
  e3.bias = h->has_bias ? h->bias1 + 3 * size_t(H) : nullptr;
  PB_CUDA(pb::launch_gemm(pb::kEpiBlockIn, h->op16, tm_xn, tm_w1, T, n_h, H, e3, h->num_sms,
                          h->status, h->limit_ns, scratch + L.sk, st),
          "MLP input GEMM launch");
  // 7. y = h + GeLU(.) W2 (+ b2): A = act[:, H:H+F], columns [H, H + F) of W2cat
  CUtensorMap tm_g, tm_w2;
  s = make_map_2d(&tm_g, act + size_t(H) * esz, T, F, H + F, box, h->op16);
  if (s == PB_OK) s = make_map_2d(&tm_w2, w2c + size_t(H) * esz, H, F, H + F, box, h->op16);
  if (s != PB_OK) return s;
  EpiParams e4{};
  e4.status = h->status;
  e4.bias = h->has_bias ? h->bias_2 : nullptr;
  e4.resid = hres;
  e4.resid_f32 = true;
  e4.y = y;
  e4.y_f32 = false;
  PB_CUDA(pb::launch_gemm(pb::kEpiResidual, h->op16, tm_g, tm_w2, T, H, F, e4, h->num_sms,
                          h->status, h->limit_ns, scratch + L.sk, st),
          "MLP output GEMM launch");
  return PB_OK;
}

// The block's backward pass (see pb_backward in pb.h) after run_block(..., train = true) on
// the same scratch. Nine steps, each on the handle's stream:
//   1. [d_attn | d act] = dy [Wo ; W2]^T (B = W2cat read MN-major), dh = d act * act'(h)
//   2. delta = d_attn . O per row and head
//   3. attention backward: dq (fp32 accumulator, then bf16), dk, dv into dz
//   4. dLN(x) = dz W1cat (B = W1cat read MN-major), fp32
//   5. dx = dy + norm'(x)^T dLN(x); dgamma, dbeta
//   6. [dWo ; dW2] = act^T dy     (both operands MN-major: the contraction runs over tokens)
//   7. [dWqkv | dW1] = LN(x)^T dz
//   8. bias gradients: column sums of dy and dz
pb_status run_backward(pb_handle* h, const void* x, const void* dy, const pb_grads& g,
                       bool acc, uint8_t* scratch, cudaStream_t st) {
  const pb_dims& d = h->d;
  const pb_scratch_layout L = scratch_layout(d);
  const int H = d.hidden, F = d.ffn, T = d.batch * d.seq;
  const bool glu = is_glu(d);
  const int NZ = int(w1_rows(d)), Fp = NZ - 3 * H;
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(scratch + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(scratch + off); };
  __nv_bfloat16 *d_attn = bf(L.d_attn), *dz = bf(L.dz);
  const uint32_t box = pb::kGemmBoxRows;
  const int big = 0x7fffffff;

  // 1. d_attn, dh
  CUtensorMap tm_dy, tm_w2t;
  pb_status s = make_map_2d(&tm_dy, dy, T, H, H, box);
  if (s == PB_OK) s = make_map_2d(&tm_w2t, h->w2cat, H, H + F, H + F, 64);
  if (s != PB_OK) return s;
  EpiParams e1{};
  e1.status = h->status;
  e1.H = H;
  e1.F = F;
  e1.glu = glu;
  e1.hpre = bf(L.hpre);
  e1.d_attn = d_attn;
  e1.dz = dz;
  e1.ldz = NZ;
  PB_CUDA(pb::launch_gemm_layout(pb::kEpiBwdAct, pb::kKM, tm_dy, tm_w2t, T, H + F, H, e1,
                                 h->num_sms, h->status, h->limit_ns, scratch + L.sk, st),
          "backward GEMM (d_attn, dh) launch");
  // 2. delta
  PB_CUDA(pb::launch_attn_delta(d_attn, bf(L.act), H + F, d.batch, d.seq, d.heads, d.head_dim,
                                f32(L.delta), int64_t(lse_ld(d)), st),
          "delta launch");
  // 3. attention backward
  CUtensorMap tm_q, tm_k, tm_vt, tm_do, tm_dq;
  {
    const uint64_t qdims[3] = {2 * uint64_t(H), uint64_t(d.seq), uint64_t(d.batch)};
    const uint64_t qstr[2] = {2 * uint64_t(H) * 2, 2 * uint64_t(H) * 2 * uint64_t(d.seq)};
    const uint32_t qbox[3] = {64, 64, 1}, kbox[3] = {64, 128, 1};
    const uint64_t odims[3] = {uint64_t(H), uint64_t(d.seq), uint64_t(d.batch)};
    const uint64_t ostr[2] = {uint64_t(H) * 2, uint64_t(H) * 2 * uint64_t(d.seq)};
    const uint64_t vdims[2] = {uint64_t(d.seq), uint64_t(d.batch) * H};
    const uint64_t vstr[1] = {uint64_t(L.seq_pad) * 2};
    const uint32_t vbox[2] = {64, uint32_t(d.head_dim)};
    s = make_map(&tm_q, scratch + L.qk, 3, qdims, qstr, qbox);
    if (s == PB_OK) s = make_map(&tm_k, scratch + L.qk, 3, qdims, qstr, kbox);
    if (s == PB_OK) s = make_map(&tm_vt, scratch + L.vt, 2, vdims, vstr, vbox);
    if (s == PB_OK) s = make_map(&tm_do, d_attn, 3, odims, ostr, qbox);
    const uint64_t fstr[2] = {uint64_t(H) * 4, uint64_t(H) * 4 * uint64_t(d.seq)};
    const uint32_t fbox[3] = {32, 64, 1};
    if (s == PB_OK) s = make_map_f32(&tm_dq, scratch + L.dq_acc, 3, odims, fstr, fbox);
    if (s != PB_OK) return s;
  }
  PB_CUDA(cudaMemsetAsync(f32(L.dq_acc), 0, size_t(T) * H * 4, st), "cudaMemsetAsync(dq)");
  pb::SwaBwdParams sb{};
  sb.B = d.batch;
  sb.S = d.seq;
  sb.H = H;
  sb.nh = d.heads;
  sb.dh = d.head_dim;
  sb.window = d.window;
  sb.scale = float(1.0 / std::sqrt(double(d.head_dim)));
  sb.scale_log2 = float(1.4426950408889634 / std::sqrt(double(d.head_dim)));
  sb.lse = f32(L.lse);
  sb.delta = f32(L.delta);
  sb.lse_ld = int64_t(lse_ld(d));
  sb.dq_acc = f32(L.dq_acc);
  sb.dz = dz;
  sb.ldz = NZ;
  PB_CUDA(pb::launch_swa_bwd(tm_q, tm_k, tm_vt, tm_do, tm_dq, sb, h->status, h->limit_ns, st),
          "attention backward launch");
  PB_CUDA(pb::launch_dq_to_bf16(f32(L.dq_acc), T, H, sb.scale, dz, NZ, st), "dq launch");
  // 4. dLN(x) = dz W1cat
  CUtensorMap tm_dz, tm_w1t;
  s = make_map_2d(&tm_dz, dz, T, NZ, NZ, box);
  if (s == PB_OK) s = make_map_2d(&tm_w1t, h->w1cat, NZ, H, H, 64);
  if (s != PB_OK) return s;
  EpiParams e4{};
  e4.status = h->status;
  e4.g0 = f32(L.dxn);
  e4.ld0 = H;
  e4.split_row = big;
  e4.split_col = big;
  PB_CUDA(pb::launch_gemm_layout(pb::kEpiGrad, pb::kKM, tm_dz, tm_w1t, T, H, NZ, e4, h->num_sms,
                                 h->status, h->limit_ns, scratch + L.sk, st),
          "backward GEMM (dLN(x)) launch");
  // 5. the normalisation and the residual
  auto* stats = reinterpret_cast<float2*>(scratch + L.stats);
  PB_CUDA(pb::launch_norm_bwd(T, H, static_cast<const __nv_bfloat16*>(x), h->gamma, f32(L.dxn),
                              static_cast<const __nv_bfloat16*>(dy), d.ln_eps, glu,
                              static_cast<__nv_bfloat16*>(g.dx), stats, st),
          "norm backward launch");
  PB_CUDA(pb::launch_norm_param_grads(T, H, static_cast<const __nv_bfloat16*>(x), f32(L.dxn),
                                      stats, f32(L.partials), g.dgamma,
                                      glu ? nullptr : g.dbeta, acc, st),
          "norm parameter gradients launch");
  // 6. [dWo ; dW2] = act^T dy
  CUtensorMap tm_act_t, tm_dy_t;
  s = make_map_2d(&tm_act_t, scratch + L.act, T, H + F, H + F, 64);
  if (s == PB_OK) s = make_map_2d(&tm_dy_t, dy, T, H, H, 64);
  if (s != PB_OK) return s;
  EpiParams e6{};
  e6.status = h->status;
  e6.g0 = g.dwo;
  e6.ld0 = H;
  e6.g1 = g.dw2;
  e6.ld1 = H;
  e6.split_row = H;
  e6.split_col = big;
  e6.accumulate = acc;
  PB_CUDA(pb::launch_gemm_layout(pb::kEpiGrad, pb::kMM, tm_act_t, tm_dy_t, H + F, H, T, e6,
                                 h->num_sms, h->status, h->limit_ns, scratch + L.sk, st),
          "weight gradient GEMM (Wo, W2) launch");
  // 7. [dWqkv | dW1] = LN(x)^T dz
  CUtensorMap tm_xn_t, tm_dz_t;
  s = make_map_2d(&tm_xn_t, scratch + L.xn, T, H, H, 64);
  if (s == PB_OK) s = make_map_2d(&tm_dz_t, dz, T, NZ, NZ, 64);
  if (s != PB_OK) return s;
  EpiParams e7{};
  e7.status = h->status;
  e7.g0 = g.dwqkv;
  e7.ld0 = 3 * H;
  e7.g1 = g.dw1;
  e7.ld1 = Fp;
  e7.split_row = big;
  e7.split_col = 3 * H;
  e7.glu = glu;
  e7.F = F;
  e7.accumulate = acc;
  PB_CUDA(pb::launch_gemm_layout(pb::kEpiGrad, pb::kMM, tm_xn_t, tm_dz_t, H, NZ, T, e7,
                                 h->num_sms, h->status, h->limit_ns, scratch + L.sk, st),
          "weight gradient GEMM (Wqkv, W1) launch");
  // 8. biases
  const auto* dyb = static_cast<const __nv_bfloat16*>(dy);
  if (g.db_o != nullptr)
    PB_CUDA(pb::launch_col_sums(dyb, T, H, H, f32(L.partials), g.db_o, nullptr, H, 0, acc, st),
            "bias gradient launch");
  if (g.db2 != nullptr)
    PB_CUDA(pb::launch_col_sums(dyb, T, H, H, f32(L.partials), g.db2, nullptr, H, 0, acc, st),
            "bias gradient launch");
  if (g.db_qkv != nullptr || g.db1 != nullptr)
    PB_CUDA(pb::launch_col_sums(dz, T, NZ, NZ, f32(L.partials), g.db_qkv, g.db1, 3 * H,
                                glu ? F : 0, acc, st),
            "bias gradient launch");
  return PB_OK;
}

pb_status check_train(pb_handle* h) {
  if (h->f16 || h->fp8)
    return fail(PB_ERR_UNSUPPORTED, "training needs PB_OPERANDS_BF16 operands");
  return PB_OK;
}

void trace_free(pb_handle* h) {
  for (cudaEvent_t e : h->trace) cudaEventDestroy(e);
  h->trace.clear();
  h->trace_max = 0;
  h->trace_calls = 0;
}

pb_status check_stack(pb_handle* const* layers, int32_t n_layers, const void* scratch,
                      size_t scratch_bytes) {
  if (layers == nullptr || n_layers < 1) return fail(PB_ERR_INVALID_ARG, "no layers");
  for (int32_t l = 0; l < n_layers; ++l) {
    pb_status s = check_handle(layers[l]);
    if (s != PB_OK) return s;
    if (std::memcmp(&layers[l]->d, &layers[0]->d, sizeof(pb_dims)) != 0)
      return fail(PB_ERR_INVALID_ARG, "layer %d has different dims from layer 0", l);
  }
  const pb_scratch_layout L = scratch_layout(layers[0]->d);
  if (scratch == nullptr || !aligned(scratch, 256))
    return fail(PB_ERR_INVALID_ARG, "scratch must be a 256-byte aligned device pointer");
  if (scratch_bytes < L.total)
    return fail(PB_ERR_WORKSPACE, "scratch has %zu bytes, %zu needed", scratch_bytes, L.total);
  return PB_OK;
}

// Layer 0 reads bf16 x, the last layer writes y (bf16, or fp32 when y_f32); in between
// the residual stream alternates between the fp32 buffers res0 and res1.
pb_status run_stack(pb_handle* const* layers, int32_t n, const void* x, void* y,
                    uint8_t* scratch, cudaStream_t st, bool y_f32 = false) {
  const pb_scratch_layout L = scratch_layout(layers[0]->d);
  void* res[2] = {scratch + L.res0, scratch + L.res1};
  const void* in = x;
  bool in_f32 = false;
  for (int32_t l = 0; l < n; ++l) {
    const bool last = (l == n - 1);
    void* out = last ? y : res[l % 2];
    pb_status s = run_block(layers[l], in, in_f32, out, !last || y_f32, scratch, st);
    if (s != PB_OK) return s;
    in = out;
    in_f32 = !last;
  }
  return PB_OK;
}

}  // namespace

namespace pb {
// Records a failure of an entry point defined in another file of the library.
pb_status record_error(pb_status s, const char* message) { return fail(s, "%s", message); }
}  // namespace pb

extern "C" {

const char* pb_status_string(pb_status s) {
  switch (s) {
    case PB_OK: return "PB_OK";
    case PB_ERR_INVALID_ARG: return "PB_ERR_INVALID_ARG";
    case PB_ERR_UNSUPPORTED: return "PB_ERR_UNSUPPORTED";
    case PB_ERR_WORKSPACE: return "PB_ERR_WORKSPACE";
    case PB_ERR_CUDA: return "PB_ERR_CUDA";
    case PB_ERR_DEVICE_TIMEOUT: return "PB_ERR_DEVICE_TIMEOUT";
    case PB_ERR_BAD_HANDLE: return "PB_ERR_BAD_HANDLE";
    case PB_ERR_RANGE: return "PB_ERR_RANGE";
  }
  return "unknown pb_status";
}

const char* pb_last_error_message(void) { return g_last_error.c_str(); }

pb_status pb_weight_workspace_bytes(const pb_dims* dims, size_t* bytes) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (bytes == nullptr) return fail(PB_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ws_layout(*dims).total;
  return PB_OK;
}

pb_status pb_scratch_bytes(const pb_dims* dims, size_t* bytes) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (bytes == nullptr) return fail(PB_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = scratch_layout(*dims).total;
  return PB_OK;
}

pb_status pb_get_scratch_layout(const pb_dims* dims, pb_scratch_layout* layout) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (layout == nullptr) return fail(PB_ERR_INVALID_ARG, "layout is NULL");
  *layout = scratch_layout(*dims);
  return PB_OK;
}

pb_status pb_create(const pb_dims* dims, const pb_weights* w, void* workspace,
                    size_t workspace_bytes, void* stream, pb_handle** out) {
  return pb_create_ex(dims, w, nullptr, workspace, workspace_bytes, stream, out);
}

pb_status pb_create_ex(const pb_dims* dims, const pb_weights* w, const pb_options* options,
                       void* workspace, size_t workspace_bytes, void* stream, pb_handle** out) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (out == nullptr) return fail(PB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (w == nullptr) return fail(PB_ERR_INVALID_ARG, "weights is NULL");
  const void* req[6] = {w->ln_gamma, w->ln_beta, w->wqkv, w->w1, w->wo, w->w2};
  const char* names[6] = {"ln_gamma", "ln_beta", "wqkv", "w1", "wo", "w2"};
  for (int i = 0; i < 6; ++i) {
    if (i == 1 && is_glu(*dims) && req[i] == nullptr) continue;  // RMSNorm has no beta
    if (req[i] == nullptr) return fail(PB_ERR_INVALID_ARG, "weights.%s is NULL", names[i]);
    if (!aligned(req[i], 16))
      return fail(PB_ERR_INVALID_ARG, "weights.%s is not 16-byte aligned", names[i]);
  }
  const void* biases[4] = {w->b_qkv, w->b1, w->b_o, w->b2};
  for (int i = 0; i < 4; ++i)
    if (biases[i] != nullptr && !aligned(biases[i], 2))
      return fail(PB_ERR_INVALID_ARG, "a bias pointer is misaligned");
  pb_options opt{PB_OPERANDS_BF16, 0};
  if (options != nullptr) opt = *options;
  if (opt.operand_precision != PB_OPERANDS_BF16 && opt.operand_precision != PB_OPERANDS_FP16 &&
      opt.operand_precision != PB_OPERANDS_FP8)
    return fail(PB_ERR_INVALID_ARG, "operand_precision %d is not a pb_operand_precision",
                opt.operand_precision);
  // FP8 GEMMs step through K in 128-element stages: K = H (first GEMM) and H + F (second)
  if (opt.operand_precision == PB_OPERANDS_FP8 &&
      (dims->hidden % pb::kGemmBK8 != 0 || (dims->hidden + dims->ffn) % pb::kGemmBK8 != 0))
    return fail(PB_ERR_UNSUPPORTED, "FP8 operands need hidden and hidden + ffn to be multiples of %d",
                pb::kGemmBK8);
  const WsLayout L = ws_layout(*dims);
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(PB_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (workspace_bytes < L.total)
    return fail(PB_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, L.total);

  int dev = -1, sms = 0;
  PB_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  PB_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
          "cudaDeviceGetAttribute");
  pb_handle* h = new (std::nothrow) pb_handle();
  if (h == nullptr) return fail(PB_ERR_INVALID_ARG, "host allocation of the handle failed");
  h->magic = kMagic;
  h->d = *dims;
  h->device = dev;
  h->num_sms = sms;
  h->limit_ns = opt.wait_limit_ns ? opt.wait_limit_ns : kDefaultLimitNs;
  h->f16 = opt.operand_precision == PB_OPERANDS_FP16;
  h->fp8 = opt.operand_precision == PB_OPERANDS_FP8;
  h->op16 = h->f16 ? pb::kOpF16 : pb::kOpBf16;
  h->gop = h->fp8 ? pb::kOpE4m3 : h->op16;
  h->ws = static_cast<uint8_t*>(workspace);
  h->status = reinterpret_cast<int*>(h->ws + L.status);
  h->w1cat = h->ws + L.w1cat;
  h->w2cat = h->ws + L.w2cat;
  h->w1scale = reinterpret_cast<float*>(h->ws + L.w1scale);
  h->w2scale = reinterpret_cast<float*>(h->ws + L.w2scale);
  h->bias1 = reinterpret_cast<float*>(h->ws + L.bias1);
  h->bias2 = reinterpret_cast<float*>(h->ws + L.bias2);
  h->bias_o = reinterpret_cast<float*>(h->ws + L.bias_o);
  h->bias_2 = reinterpret_cast<float*>(h->ws + L.bias_2);
  h->gamma = reinterpret_cast<__nv_bfloat16*>(h->ws + L.gamma);
  h->beta = reinterpret_cast<__nv_bfloat16*>(h->ws + L.beta);
  h->has_bias = w->b_qkv || w->b1 || w->b_o || w->b2;

  const int64_t H = dims->hidden, F = dims->ffn;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto bf = [](const void* p) { return static_cast<const __nv_bfloat16*>(p); };
  auto cleanup = [&](pb_status e) {
    h->magic = kDead;
    delete h;
    return e;
  };
#define PB_CUDA_H(call, what)                                \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cleanup(cuda_fail(e_, what)); \
  } while (0)
  PB_CUDA_H(cudaMemsetAsync(h->status, 0, 256, st), "cudaMemsetAsync(status)");
  // W1cat rows [0, 3H) = Wqkv^T, rows [3H, 3H + F) = W1^T (SwiGLU: rows [3H, 3H + 2F) =
  // [W_gate | W_up]^T interleaved in groups of 16)
  const bool glu = is_glu(*dims);
  const int64_t w1_cols = glu ? 2 * F : F;
  uint8_t* w1c = static_cast<uint8_t*>(h->w1cat);
  uint8_t* w2c = static_cast<uint8_t*>(h->w2cat);
  if (h->fp8) {
    // E4M3 codes with one scale per output channel (amax / 448): the channel's amax over
    // the columns of Wqkv and W1 (source order), and over Wo's and W2's columns together
    float* amax1 = reinterpret_cast<float*>(h->ws + L.amax1);
    float* amax2 = reinterpret_cast<float*>(h->ws + L.amax2);
    PB_CUDA_H(cudaMemsetAsync(amax1, 0, size_t(w1_rows(*dims)) * 4, st), "cudaMemsetAsync(amax)");
    PB_CUDA_H(cudaMemsetAsync(amax2, 0, size_t(H) * 4, st), "cudaMemsetAsync(amax)");
    PB_CUDA_H(pb::launch_col_amax(bf(w->wqkv), H, 3 * H, 3 * H, amax1, st), "amax of Wqkv");
    PB_CUDA_H(pb::launch_col_amax(bf(w->w1), H, w1_cols, w1_cols, amax1 + 3 * H, st),
              "amax of W1");
    PB_CUDA_H(pb::launch_col_amax(bf(w->wo), H, H, H, amax2, st), "amax of Wo");
    PB_CUDA_H(pb::launch_col_amax(bf(w->w2), F, H, H, amax2, st), "amax of W2");
    PB_CUDA_H(pb::launch_transpose_e4m3(bf(w->wqkv), H, 3 * H, 3 * H, w1c, H, 0, amax1, st),
              "pack Wqkv");
    PB_CUDA_H(pb::launch_transpose_e4m3(bf(w->w1), H, w1_cols, w1_cols, w1c + 3 * H * H, H,
                                        glu ? F : 0, amax1 + 3 * H, st),
              "pack W1");
    PB_CUDA_H(pb::launch_transpose_e4m3(bf(w->wo), H, H, H, w2c, H + F, 0, amax2, st), "pack Wo");
    PB_CUDA_H(pb::launch_transpose_e4m3(bf(w->w2), F, H, H, w2c + H, H + F, 0, amax2, st),
              "pack W2");
    PB_CUDA_H(pb::launch_amax_to_scales(amax1, 3 * H, 0, h->w1scale, st), "W1cat scales");
    PB_CUDA_H(pb::launch_amax_to_scales(amax1 + 3 * H, w1_cols, glu ? F : 0, h->w1scale + 3 * H,
                                        st),
              "W1cat scales");
    PB_CUDA_H(pb::launch_amax_to_scales(amax2, H, 0, h->w2scale, st), "W2cat scales");
  } else {
    PB_CUDA_H(pb::launch_transpose(bf(w->wqkv), H, 3 * H, 3 * H, w1c, H, h->f16, 0, h->status, st),
              "pack Wqkv");
    PB_CUDA_H(pb::launch_transpose(bf(w->w1), H, w1_cols, w1_cols, w1c + 3 * H * H * 2, H, h->f16,
                                   glu ? F : 0, h->status, st),
              "pack W1");
    // W2cat columns [0, H) = Wo^T, columns [H, H + F) = W2^T
    PB_CUDA_H(pb::launch_transpose(bf(w->wo), H, H, H, w2c, H + F, h->f16, 0, h->status, st),
              "pack Wo");
    PB_CUDA_H(pb::launch_transpose(bf(w->w2), F, H, H, w2c + H * 2, H + F, h->f16, 0, h->status,
                                   st),
              "pack W2");
  }
  PB_CUDA_H(pb::launch_bias_prep(bf(w->b_qkv), bf(w->b1), bf(w->b_o), bf(w->b2), int(H), int(F),
                                 glu, h->bias1, h->bias2, h->bias_o, h->bias_2, st),
            "bias prep");
  PB_CUDA_H(cudaMemcpyAsync(h->gamma, w->ln_gamma, H * 2, cudaMemcpyDeviceToDevice, st),
            "copy gamma");
  if (w->ln_beta != nullptr)
    PB_CUDA_H(cudaMemcpyAsync(h->beta, w->ln_beta, H * 2, cudaMemcpyDeviceToDevice, st),
              "copy beta");
#undef PB_CUDA_H
  s = make_map_2d(&h->tm_w1cat, h->w1cat, w1_rows(*dims), H, H, pb::kGemmBoxRows, h->gop);
  if (s == PB_OK)
    s = make_map_2d(&h->tm_w2cat, h->w2cat, H, H + F, H + F, pb::kGemmBoxRows, h->gop);
  if (s != PB_OK) return cleanup(s);
  *out = h;
  return PB_OK;
}

pb_status pb_forward(pb_handle* h, const void* x, void* y, void* scratch, size_t scratch_bytes,
                     void* stream) {
  pb_status s = check_stack(&h, 1, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
    return fail(PB_ERR_INVALID_ARG, "x and y must be 16-byte aligned device pointers");
  const size_t n = size_t(h->d.batch) * h->d.seq * h->d.hidden * 2;
  if (x != y && overlap(x, n, y, n))
    return fail(PB_ERR_INVALID_ARG, "x and y overlap without being equal");
  const pb_scratch_layout L = scratch_layout(h->d);
  if (overlap(x, n, scratch, L.total) || overlap(y, n, scratch, L.total))
    return fail(PB_ERR_INVALID_ARG, "x or y overlaps the scratch buffer");
  return run_block(h, x, false, y, false, static_cast<uint8_t*>(scratch),
                   static_cast<cudaStream_t>(stream));
}

pb_status pb_train_scratch_bytes(const pb_dims* dims, size_t* bytes) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (bytes == nullptr) return fail(PB_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = scratch_layout(*dims).train_total;
  return PB_OK;
}

pb_status pb_forward_train(pb_handle* h, const void* x, void* y, void* scratch,
                           size_t scratch_bytes, void* stream) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  s = check_train(h);
  if (s != PB_OK) return s;
  const pb_scratch_layout L = scratch_layout(h->d);
  if (scratch == nullptr || !aligned(scratch, 256))
    return fail(PB_ERR_INVALID_ARG, "scratch must be a 256-byte aligned device pointer");
  if (scratch_bytes < L.train_total)
    return fail(PB_ERR_WORKSPACE, "training scratch has %zu bytes, %zu needed", scratch_bytes,
                L.train_total);
  if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
    return fail(PB_ERR_INVALID_ARG, "x and y must be 16-byte aligned device pointers");
  const size_t n = size_t(h->d.batch) * h->d.seq * h->d.hidden * 2;
  if (x == y) return fail(PB_ERR_INVALID_ARG, "the backward reads x: y must not be x");
  if (overlap(x, n, y, n)) return fail(PB_ERR_INVALID_ARG, "x and y overlap");
  if (overlap(x, n, scratch, L.train_total) || overlap(y, n, scratch, L.train_total))
    return fail(PB_ERR_INVALID_ARG, "x or y overlaps the scratch buffer");
  return run_block(h, x, false, y, false, static_cast<uint8_t*>(scratch),
                   static_cast<cudaStream_t>(stream), true);
}

pb_status pb_backward(pb_handle* h, const void* x, const void* dy, const pb_grads* grads,
                      int32_t accumulate, void* scratch, size_t scratch_bytes, void* stream) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  s = check_train(h);
  if (s != PB_OK) return s;
  const pb_scratch_layout L = scratch_layout(h->d);
  if (scratch == nullptr || !aligned(scratch, 256))
    return fail(PB_ERR_INVALID_ARG, "scratch must be a 256-byte aligned device pointer");
  if (scratch_bytes < L.train_total)
    return fail(PB_ERR_WORKSPACE, "training scratch has %zu bytes, %zu needed", scratch_bytes,
                L.train_total);
  if (grads == nullptr) return fail(PB_ERR_INVALID_ARG, "grads is NULL");
  const void* need[7] = {x, dy, grads->dx, grads->dgamma, grads->dwqkv, grads->dw1, grads->dwo};
  for (const void* p : need)
    if (p == nullptr || !aligned(p, 16))
      return fail(PB_ERR_INVALID_ARG,
                  "x, dy, dx, dgamma and the weight gradients must be 16-byte aligned device "
                  "pointers");
  if (grads->dw2 == nullptr || !aligned(grads->dw2, 16))
    return fail(PB_ERR_INVALID_ARG, "dw2 must be a 16-byte aligned device pointer");
  const pb_dims& d = h->d;
  const size_t n = size_t(d.batch) * d.seq * d.hidden * 2;
  if (overlap(grads->dx, n, x, n) || overlap(grads->dx, n, dy, n))
    return fail(PB_ERR_INVALID_ARG, "dx overlaps x or dy");
  if (overlap(grads->dx, n, scratch, L.train_total) || overlap(dy, n, scratch, L.train_total))
    return fail(PB_ERR_INVALID_ARG, "dx or dy overlaps the scratch buffer");
  return run_backward(h, x, dy, *grads, accumulate != 0, static_cast<uint8_t*>(scratch),
                      static_cast<cudaStream_t>(stream));
}

pb_status pb_forward_serial(pb_handle* h, const void* x, void* y, const void* ln2_gamma,
                            const void* ln2_beta, void* scratch, size_t scratch_bytes,
                            void* stream) {
  pb_status s = check_stack(&h, 1, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (h->fp8) return fail(PB_ERR_UNSUPPORTED, "pb_forward_serial does not take FP8 operands");
  if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
    return fail(PB_ERR_INVALID_ARG, "x and y must be 16-byte aligned device pointers");
  if ((ln2_gamma == nullptr) != (ln2_beta == nullptr))
    return fail(PB_ERR_INVALID_ARG, "ln2_gamma and ln2_beta must both be given or both NULL");
  if ((ln2_gamma != nullptr && !aligned(ln2_gamma, 16)) ||
      (ln2_beta != nullptr && !aligned(ln2_beta, 16)))
    return fail(PB_ERR_INVALID_ARG, "ln2_gamma and ln2_beta must be 16-byte aligned");
  const size_t n = size_t(h->d.batch) * h->d.seq * h->d.hidden * 2;
  if (x != y && overlap(x, n, y, n))
    return fail(PB_ERR_INVALID_ARG, "x and y overlap without being equal");
  const pb_scratch_layout L = scratch_layout(h->d);
  if (overlap(x, n, scratch, L.total) || overlap(y, n, scratch, L.total))
    return fail(PB_ERR_INVALID_ARG, "x or y overlaps the scratch buffer");
  const auto* g2 = ln2_gamma ? static_cast<const __nv_bfloat16*>(ln2_gamma) : h->gamma;
  const auto* b2 = ln2_beta ? static_cast<const __nv_bfloat16*>(ln2_beta) : h->beta;  // unused by RMSNorm
  return run_serial(h, x, y, g2, b2, static_cast<uint8_t*>(scratch),
                    static_cast<cudaStream_t>(stream));
}

pb_status pb_forward_stack(pb_handle* const* layers, int32_t n_layers, const void* x, void* y,
                           void* scratch, size_t scratch_bytes, void* stream) {
  pb_status s = check_stack(layers, n_layers, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
    return fail(PB_ERR_INVALID_ARG, "x and y must be 16-byte aligned device pointers");
  const pb_dims& d = layers[0]->d;
  const size_t n = size_t(d.batch) * d.seq * d.hidden * 2;
  if (x != y && overlap(x, n, y, n))
    return fail(PB_ERR_INVALID_ARG, "x and y overlap without being equal");
  const pb_scratch_layout L = scratch_layout(d);
  if (overlap(x, n, scratch, L.total) || overlap(y, n, scratch, L.total))
    return fail(PB_ERR_INVALID_ARG, "x or y overlaps the scratch buffer");
  return run_stack(layers, n_layers, x, y, static_cast<uint8_t*>(scratch),
                   static_cast<cudaStream_t>(stream));
}

pb_status pb_forward_stack_f32(pb_handle* const* layers, int32_t n_layers, const void* x,
                               float* y, void* scratch, size_t scratch_bytes, void* stream) {
  pb_status s = check_stack(layers, n_layers, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (x == nullptr || y == nullptr || !aligned(x, 16) || !aligned(y, 16))
    return fail(PB_ERR_INVALID_ARG, "x and y must be 16-byte aligned device pointers");
  const pb_dims& d = layers[0]->d;
  const size_t nx = size_t(d.batch) * d.seq * d.hidden * 2, ny = 2 * nx;
  if (overlap(x, nx, y, ny)) return fail(PB_ERR_INVALID_ARG, "x and y overlap");
  const pb_scratch_layout L = scratch_layout(d);
  if (overlap(x, nx, scratch, L.total) || overlap(y, ny, scratch, L.total))
    return fail(PB_ERR_INVALID_ARG, "x or y overlaps the scratch buffer");
  return run_stack(layers, n_layers, x, y, static_cast<uint8_t*>(scratch),
                   static_cast<cudaStream_t>(stream), true);
}

pb_status pb_forward_stack_host(pb_handle* const* layers, int32_t n_layers, const void* x_host,
                                void* y_host, void* scratch, size_t scratch_bytes, void* stream) {
  pb_status s = check_stack(layers, n_layers, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (x_host == nullptr || y_host == nullptr)
    return fail(PB_ERR_INVALID_ARG, "x_host and y_host must be host pointers");
  const pb_dims& d = layers[0]->d;
  const size_t n = size_t(d.batch) * d.seq * d.hidden * 2;
  const pb_scratch_layout L = scratch_layout(d);
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  void* io = sc + L.io;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PB_CUDA(cudaMemcpyAsync(io, x_host, n, cudaMemcpyHostToDevice, st), "copy x to the device");
  // io holds x for layer 0 and receives y from the last layer (in place when there is one
  // layer; later layers no longer read x).
  s = run_stack(layers, n_layers, io, io, sc, st);
  if (s != PB_OK) return s;
  PB_CUDA(cudaMemcpyAsync(y_host, io, n, cudaMemcpyDeviceToHost, st), "copy y to the host");
  return PB_OK;
}

pb_status pb_forward_stack_host_steps(pb_handle* const* layers, int32_t n_layers,
                                      int32_t n_steps, const void* const* x_host,
                                      void* const* y_host, void* scratch, size_t scratch_bytes,
                                      void* stream) {
  pb_status s = check_stack(layers, n_layers, scratch, scratch_bytes);
  if (s != PB_OK) return s;
  if (n_steps < 1 || x_host == nullptr || y_host == nullptr)
    return fail(PB_ERR_INVALID_ARG, "need n_steps >= 1 and arrays of host pointers");
  for (int32_t i = 0; i < n_steps; ++i)
    if (x_host[i] == nullptr || y_host[i] == nullptr)
      return fail(PB_ERR_INVALID_ARG, "x_host[%d] or y_host[%d] is NULL", i, i);
  pb_handle* h0 = layers[0];
  if (h0->copy_stream == nullptr) {
    PB_CUDA(cudaStreamCreateWithFlags(&h0->copy_stream, cudaStreamNonBlocking),
            "cudaStreamCreateWithFlags");
    for (cudaEvent_t& e : h0->copy_ev)
      PB_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
  }
  const pb_dims& d = h0->d;
  const size_t n = size_t(d.batch) * d.seq * d.hidden * 2;
  const pb_scratch_layout L = scratch_layout(d);
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  void* io[2] = {sc + L.io, sc + L.io2};
  cudaStream_t st = static_cast<cudaStream_t>(stream), cs = h0->copy_stream;
  cudaEvent_t ev_start = h0->copy_ev[0], ev_out = h0->copy_ev[5];
  cudaEvent_t ev_in[2] = {h0->copy_ev[1], h0->copy_ev[2]};
  cudaEvent_t ev_done[2] = {h0->copy_ev[3], h0->copy_ev[4]};
  // The copy stream starts after the work already queued on `stream` (which may use io).
  // Its order is H2D(0), H2D(1), D2H(0), H2D(2), D2H(1), ...: the input of step s + 1 and
  // the output of step s - 1 move while step s computes; an io buffer is refilled only
  // after its previous output has been copied out (the copy stream is in order).
  PB_CUDA(cudaEventRecord(ev_start, st), "cudaEventRecord");
  PB_CUDA(cudaStreamWaitEvent(cs, ev_start, 0), "cudaStreamWaitEvent");
  PB_CUDA(cudaMemcpyAsync(io[0], x_host[0], n, cudaMemcpyHostToDevice, cs), "copy x");
  PB_CUDA(cudaEventRecord(ev_in[0], cs), "cudaEventRecord");
  for (int32_t i = 0; i < n_steps; ++i) {
    const int b = i & 1;
    PB_CUDA(cudaStreamWaitEvent(st, ev_in[b], 0), "cudaStreamWaitEvent");
    s = run_stack(layers, n_layers, io[b], io[b], sc, st);
    if (s != PB_OK) return s;
    PB_CUDA(cudaEventRecord(ev_done[b], st), "cudaEventRecord");
    if (i + 1 < n_steps) {
      PB_CUDA(cudaMemcpyAsync(io[b ^ 1], x_host[i + 1], n, cudaMemcpyHostToDevice, cs),
              "copy x");
      PB_CUDA(cudaEventRecord(ev_in[b ^ 1], cs), "cudaEventRecord");
    }
    PB_CUDA(cudaStreamWaitEvent(cs, ev_done[b], 0), "cudaStreamWaitEvent");
    PB_CUDA(cudaMemcpyAsync(y_host[i], io[b], n, cudaMemcpyDeviceToHost, cs), "copy y");
  }
  // `stream` reaches the point after this call only when every output is on the host
  PB_CUDA(cudaEventRecord(ev_out, cs), "cudaEventRecord");
  PB_CUDA(cudaStreamWaitEvent(st, ev_out, 0), "cudaStreamWaitEvent");
  return PB_OK;
}

pb_status pb_get_status(pb_handle* h) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  int word = 0;
  PB_CUDA(cudaMemcpy(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost), "read status word");
  if (word == 0) return PB_OK;
  return fail(pb_status(word & 0xff), "device status word 0x%x (wait site %d)", word, word >> 8);
}

pb_status pb_clear_status(pb_handle* h, void* stream) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  PB_CUDA(cudaMemsetAsync(h->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)),
          "clear status word");
  return PB_OK;
}

pb_status pb_set_wait_limit_ns(pb_handle* h, uint64_t limit_ns) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  if (limit_ns == 0) return fail(PB_ERR_INVALID_ARG, "limit must be > 0");
  h->limit_ns = limit_ns;
  return PB_OK;
}

pb_status pb_trace_enable(pb_handle* h, int32_t n_calls) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  if (n_calls < 0 || n_calls > (1 << 20)) return fail(PB_ERR_INVALID_ARG, "n_calls out of range");
  trace_free(h);
  h->trace.resize(size_t(n_calls) * 5, nullptr);
  for (auto& e : h->trace) {
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) {
      e = nullptr;
      for (auto& f : h->trace)
        if (f) cudaEventDestroy(f);
      h->trace.clear();
      return cuda_fail(err, "cudaEventCreate");
    }
  }
  h->trace_max = n_calls;
  return PB_OK;
}

pb_status pb_trace_read(pb_handle* h, float* ms, int32_t* calls) {
  pb_status s = check_handle(h);
  if (s != PB_OK) return s;
  if (ms == nullptr || calls == nullptr) return fail(PB_ERR_INVALID_ARG, "ms or calls is NULL");
  for (int k = 0; k < 4; ++k) ms[k] = 0.f;
  for (int c = 0; c < h->trace_calls; ++c) {
    cudaEvent_t* ev = &h->trace[size_t(c) * 5];
    PB_CUDA(cudaEventSynchronize(ev[4]), "cudaEventSynchronize");
    for (int k = 0; k < 4; ++k) {
      float t = 0.f;
      PB_CUDA(cudaEventElapsedTime(&t, ev[k], ev[k + 1]), "cudaEventElapsedTime");
      ms[k] += t;
    }
  }
  *calls = h->trace_calls;
  return PB_OK;
}

pb_status pb_destroy(pb_handle* h) {
  if (h == nullptr) return fail(PB_ERR_BAD_HANDLE, "handle is NULL");
  if (h->magic != kMagic) return fail(PB_ERR_BAD_HANDLE, "handle is destroyed or invalid");
  trace_free(h);
  if (h->copy_stream != nullptr) {
    cudaStreamSynchronize(h->copy_stream);
    for (cudaEvent_t e : h->copy_ev) cudaEventDestroy(e);
    cudaStreamDestroy(h->copy_stream);
  }
  h->magic = kDead;
  delete h;
  return PB_OK;
}

pb_status pb_layernorm(int64_t rows, int32_t H, const void* x, const void* gamma,
                       const void* beta, float eps, void* out, void* stream) {
  if (rows < 0 || H < 8 || H % 8 != 0 || H > pb::kLnMaxH)
    return fail(PB_ERR_UNSUPPORTED, "layernorm needs rows >= 0, H % 8 == 0, 8 <= H <= %d",
                pb::kLnMaxH);
  if (rows >= (int64_t(1) << 31)) return fail(PB_ERR_UNSUPPORTED, "rows >= 2^31");
  if (!(eps > 0.f)) return fail(PB_ERR_INVALID_ARG, "eps must be > 0");
  const void* ps[3] = {x, gamma, out};
  for (const void* p : ps)
    if (p == nullptr || !aligned(p, 16))
      return fail(PB_ERR_INVALID_ARG, "pointers must be 16-byte aligned device pointers");
  if (beta != nullptr && !aligned(beta, 16))
    return fail(PB_ERR_INVALID_ARG, "beta must be 16-byte aligned (or NULL for RMSNorm)");
  PB_CUDA(pb::launch_layernorm(rows, H, x, false, static_cast<const __nv_bfloat16*>(gamma),
                               static_cast<const __nv_bfloat16*>(beta), eps, out, false, nullptr,
                               static_cast<cudaStream_t>(stream)),
          "layernorm launch");
  return PB_OK;
}

pb_status pb_quantize_rows_e4m3(int64_t rows, int32_t cols, const void* x, void* codes,
                                void* scales, void* stream) {
  if (rows < 0 || cols < 8 || cols % 8 != 0)
    return fail(PB_ERR_UNSUPPORTED, "quantize needs rows >= 0 and cols %% 8 == 0, cols >= 8");
  if (rows >= (int64_t(1) << 31)) return fail(PB_ERR_UNSUPPORTED, "rows >= 2^31");
  const void* ps[3] = {x, codes, scales};
  for (const void* p : ps)
    if (p == nullptr || !aligned(p, 16))
      return fail(PB_ERR_INVALID_ARG, "pointers must be 16-byte aligned device pointers");
  PB_CUDA(pb::launch_quantize_rows_e4m3(static_cast<const __nv_bfloat16*>(x), rows, cols, cols,
                                        static_cast<uint8_t*>(codes), cols,
                                        static_cast<float*>(scales),
                                        static_cast<cudaStream_t>(stream)),
          "quantize launch");
  return PB_OK;
}

pb_status pb_set_guard_bytes(size_t bytes) {
  if (bytes > (size_t(1) << 20)) return fail(PB_ERR_INVALID_ARG, "guard of %zu bytes > 1 MiB", bytes);
  g_guard_bytes.store(bytes, std::memory_order_relaxed);
  return PB_OK;
}

pb_status pb_get_guard_bytes(size_t* bytes) {
  if (bytes == nullptr) return fail(PB_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = g_guard_bytes.load(std::memory_order_relaxed);
  return PB_OK;
}

pb_status pb_gemm_scratch_bytes(size_t* bytes) {
  if (bytes == nullptr) return fail(PB_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = pb::kSkScratchBytes;
  return PB_OK;
}

pb_status pb_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, const void* B, void* C,
                       void* scratch, size_t scratch_bytes, int* status, void* stream) {
  if (M < 1 || N < 1 || K < 1) return fail(PB_ERR_INVALID_ARG, "M, N, K must be >= 1");
  if (K % 64 != 0 || N % 32 != 0)
    return fail(PB_ERR_UNSUPPORTED, "gemm needs K %% 64 == 0 and N %% 32 == 0");
  if (A == nullptr || B == nullptr || C == nullptr || !aligned(A, 16) || !aligned(B, 16) ||
      !aligned(C, 16))
    return fail(PB_ERR_INVALID_ARG, "A, B, C must be 16-byte aligned device pointers");
  if (scratch != nullptr && (!aligned(scratch, 256) || scratch_bytes < pb::kSkScratchBytes))
    return fail(PB_ERR_WORKSPACE, "scratch must be NULL or 256-byte aligned with >= %zu bytes",
                pb::kSkScratchBytes);
  int dev = -1, sms = 0;
  PB_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  PB_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
          "cudaDeviceGetAttribute");
  CUtensorMap ta, tb;
  pb_status s = make_map_2d(&ta, A, uint64_t(M), uint64_t(K), uint64_t(K), pb::kGemmBoxRows);
  if (s == PB_OK) s = make_map_2d(&tb, B, uint64_t(N), uint64_t(K), uint64_t(K), pb::kGemmBoxRows);
  if (s != PB_OK) return s;
  EpiParams ep{};
  ep.c = static_cast<__nv_bfloat16*>(C);
  ep.ldc = N;
  PB_CUDA(pb::launch_gemm(pb::kEpiStore, pb::kOpBf16, ta, tb, M, N, K, ep, sms, status, kDefaultLimitNs,
                          scratch, static_cast<cudaStream_t>(stream)),
          "gemm launch");
  return PB_OK;
}

pb_status pb_gemm_bf16_layout(int32_t M, int32_t N, int32_t K, const void* A, int32_t a_mn,
                              const void* B, int32_t b_mn, void* C, void* scratch,
                              size_t scratch_bytes, int* status, void* stream) {
  if (M < 1 || N < 1 || K < 1) return fail(PB_ERR_INVALID_ARG, "M, N, K must be >= 1");
  if (N % 32 != 0) return fail(PB_ERR_UNSUPPORTED, "gemm needs N %% 32 == 0");
  if ((!a_mn || !b_mn) && K % 8 != 0)
    return fail(PB_ERR_UNSUPPORTED, "a K-major operand needs K %% 8 == 0");
  if ((a_mn && M % 8 != 0) || (b_mn && N % 8 != 0))
    return fail(PB_ERR_UNSUPPORTED, "an MN-major operand needs M (or N) %% 8 == 0");
  if (A == nullptr || B == nullptr || C == nullptr || !aligned(A, 16) || !aligned(B, 16) ||
      !aligned(C, 16))
    return fail(PB_ERR_INVALID_ARG, "A, B, C must be 16-byte aligned device pointers");
  if (scratch != nullptr && (!aligned(scratch, 256) || scratch_bytes < pb::kSkScratchBytes))
    return fail(PB_ERR_WORKSPACE, "scratch must be NULL or 256-byte aligned with >= %zu bytes",
                pb::kSkScratchBytes);
  int dev = -1, sms = 0;
  PB_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  PB_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
          "cudaDeviceGetAttribute");
  CUtensorMap ta, tb;
  pb_status s = a_mn ? make_map_2d(&ta, A, uint64_t(K), uint64_t(M), uint64_t(M), 64)
                     : make_map_2d(&ta, A, uint64_t(M), uint64_t(K), uint64_t(K), pb::kGemmBoxRows);
  if (s == PB_OK)
    s = b_mn ? make_map_2d(&tb, B, uint64_t(K), uint64_t(N), uint64_t(N), 64)
             : make_map_2d(&tb, B, uint64_t(N), uint64_t(K), uint64_t(K), pb::kGemmBoxRows);
  if (s != PB_OK) return s;
  EpiParams ep{};
  ep.c = static_cast<__nv_bfloat16*>(C);
  ep.ldc = N;
  const pb::GemmLayout layout = pb::GemmLayout((a_mn ? pb::kMK : 0) | (b_mn ? pb::kKM : 0));
  PB_CUDA(pb::launch_gemm_layout(pb::kEpiStore, layout, ta, tb, M, N, K, ep, sms, status,
                                 kDefaultLimitNs, scratch, static_cast<cudaStream_t>(stream)),
          "gemm launch");
  return PB_OK;
}

pb_status pb_swa_attention(const pb_dims* dims, const void* qk, const void* vt, void* act,
                           int64_t act_ld, int* status, void* stream) {
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  const pb_dims& d = *dims;
  if (qk == nullptr || vt == nullptr || act == nullptr || !aligned(qk, 16) || !aligned(vt, 16) ||
      !aligned(act, 16))
    return fail(PB_ERR_INVALID_ARG, "qk, vt, act must be 16-byte aligned device pointers");
  if (act_ld < d.hidden || act_ld % 8 != 0)
    return fail(PB_ERR_INVALID_ARG, "act_ld must be >= hidden and a multiple of 8");
  const int H = d.hidden;
  const size_t seq_pad = align_up(size_t(d.seq), 8);
  CUtensorMap tm_qk, tm_k, tm_vt;
  s = make_swa_maps(d, qk, vt, seq_pad, &tm_qk, &tm_k, &tm_vt);
  if (s != PB_OK) return s;
  pb::SwaParams sp{};
  sp.B = d.batch;
  sp.S = d.seq;
  sp.H = H;
  sp.nh = d.heads;
  sp.dh = d.head_dim;
  sp.window = d.window;
  sp.num_q_tiles = (d.seq + pb::kSwaBQ - 1) / pb::kSwaBQ;
  sp.scale_log2 = float(1.4426950408889634 / std::sqrt(double(d.head_dim)));
  sp.out = act;
  sp.out_ld = act_ld;
  sp.out_f16 = false;
  PB_CUDA(pb::launch_swa(tm_qk, tm_k, tm_vt, sp, status, kDefaultLimitNs,
                         static_cast<cudaStream_t>(stream)),
          "attention launch");
  return PB_OK;
}

pb_status pb_wait_probe(uint64_t limit_ns, int* status, void* stream) {
  if (status == nullptr || !aligned(status, 4))
    return fail(PB_ERR_INVALID_ARG, "status must be a 4-byte aligned device pointer");
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(PB_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
  PB_CUDA(pb::launch_wait_probe(limit_ns, status, static_cast<cudaStream_t>(stream)),
          "wait probe launch");
  return PB_OK;
}

}  // extern "C"
