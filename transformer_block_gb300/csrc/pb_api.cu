// pb_api.cu — the C ABI (include/pb.h): argument checks, workspace and scratch layout,
// TMA tensor maps, and the launch sequence of one parallel block
//   LN -> GEMM [Wqkv | W1] (+GeLU) -> sliding-window attention -> GEMM [Wo ; W2] (+x)
// (MegaScale reading notes, section 1.1, eq. (4)). All device memory belongs to the
// caller; this file allocates none.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

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
  __nv_bfloat16* w1cat;    // [3H + F, H]
  __nv_bfloat16* w2cat;    // [H, H + F]
  float* bias1;            // [3H + F]
  float* bias2;            // [H]
  __nv_bfloat16* gamma;    // [H]
  __nv_bfloat16* beta;     // [H]
  bool has_bias;
  CUtensorMap tm_w1cat;
  CUtensorMap tm_w2cat;
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
  if (int64_t(3) * d->hidden + d->ffn >= (int64_t(1) << 31))
    return fail(PB_ERR_UNSUPPORTED, "3 * hidden + ffn >= 2^31");
  return PB_OK;
}

struct WsLayout {
  size_t status, w1cat, w2cat, bias1, bias2, gamma, beta, total;
};

WsLayout ws_layout(const pb_dims& d) {
  const size_t H = size_t(d.hidden), F = size_t(d.ffn);
  WsLayout L{};
  size_t off = 0;
  L.status = off;
  off = align_up(off + 256, 1024);
  L.w1cat = off;
  off = align_up(off + (3 * H + F) * H * 2, 1024);
  L.w2cat = off;
  off = align_up(off + H * (H + F) * 2, 1024);
  L.bias1 = off;
  off = align_up(off + (3 * H + F) * 4, 1024);
  L.bias2 = off;
  off = align_up(off + H * 4, 1024);
  L.gamma = off;
  off = align_up(off + H * 2, 1024);
  L.beta = off;
  off = align_up(off + H * 2, 1024);
  L.total = off;
  return L;
}

pb_scratch_layout scratch_layout(const pb_dims& d) {
  const size_t H = size_t(d.hidden), F = size_t(d.ffn);
  const size_t T = size_t(d.batch) * size_t(d.seq);
  pb_scratch_layout L{};
  L.seq_pad = align_up(size_t(d.seq), 8);
  size_t off = 0;
  L.xn = off;
  off = align_up(off + T * H * 2, 1024);
  L.qk = off;
  off = align_up(off + T * 2 * H * 2, 1024);
  L.vt = off;
  off = align_up(off + size_t(d.batch) * H * L.seq_pad * 2, 1024);
  L.act = off;
  off = align_up(off + T * (H + F) * 2, 1024);
  L.io0 = off;
  off = align_up(off + T * H * 2, 1024);
  L.io1 = off;
  off = align_up(off + T * H * 2, 1024);
  L.total = off;
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

// bf16 tensor of `rank` dims (dims[0] innermost), 128-byte swizzle, zero fill outside.
pb_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
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
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank), const_cast<void*>(base),
                   gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PB_OK;
}

// Row-major [rows, cols] bf16 matrix read in boxes of 64 columns x box_rows rows.
pb_status make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint64_t ld, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {ld * 2};
  const uint32_t box[2] = {64, box_rows};
  return make_map(m, base, 2, dims, strides, box);
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

// One block from x to y, intermediates in `scratch`.
pb_status run_block(pb_handle* h, const __nv_bfloat16* x, __nv_bfloat16* y, uint8_t* scratch,
                    cudaStream_t st) {
  const pb_dims& d = h->d;
  const pb_scratch_layout L = scratch_layout(d);
  const int H = d.hidden, F = d.ffn, T = d.batch * d.seq;
  auto* xn = reinterpret_cast<__nv_bfloat16*>(scratch + L.xn);
  auto* qk = reinterpret_cast<__nv_bfloat16*>(scratch + L.qk);
  auto* vt = reinterpret_cast<__nv_bfloat16*>(scratch + L.vt);
  auto* act = reinterpret_cast<__nv_bfloat16*>(scratch + L.act);

  // 1. the shared LayerNorm
  PB_CUDA(pb::launch_layernorm(T, H, x, h->gamma, h->beta, d.ln_eps, xn, st), "layernorm launch");

  // 2. [q | k | v | h] = xn [Wqkv | W1], GeLU(h) in the epilogue
  CUtensorMap tm_xn, tm_act, tm_qk, tm_vt;
  pb_status s = make_map_2d(&tm_xn, xn, T, H, H, pb::kGemmBM);
  if (s != PB_OK) return s;
  EpiParams e1{};
  e1.H = H;
  e1.F = F;
  e1.S = d.seq;
  e1.nh = d.heads;
  e1.dh = d.head_dim;
  e1.seq_pad = int64_t(L.seq_pad);
  e1.qk = qk;
  e1.vt = vt;
  e1.act = act;
  e1.bias = h->has_bias ? h->bias1 : nullptr;
  PB_CUDA(pb::launch_gemm(pb::kEpiBlockIn, tm_xn, h->tm_w1cat, T, 3 * H + F, H, e1, h->num_sms,
                          h->status, h->limit_ns, st),
          "first GEMM launch");

  // 3. sliding-window attention -> act[:, 0:H]
  {
    const uint64_t dims[3] = {uint64_t(2 * H), uint64_t(d.seq), uint64_t(d.batch)};
    const uint64_t strides[2] = {uint64_t(2 * H) * 2, uint64_t(2 * H) * 2 * uint64_t(d.seq)};
    const uint32_t box[3] = {64, uint32_t(pb::kSwaBQ), 1};
    s = make_map(&tm_qk, qk, 3, dims, strides, box);
    if (s != PB_OK) return s;
    const uint64_t rows = uint64_t(d.batch) * uint64_t(H);
    const uint64_t vdims[2] = {uint64_t(d.seq), rows};
    const uint64_t vstr[1] = {uint64_t(L.seq_pad) * 2};
    const uint32_t vbox[2] = {64, uint32_t(d.head_dim)};
    s = make_map(&tm_vt, vt, 2, vdims, vstr, vbox);
    if (s != PB_OK) return s;
  }
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
  PB_CUDA(pb::launch_swa(tm_qk, tm_vt, sp, h->status, h->limit_ns, st), "attention launch");

  // 4. y = x + [attn | GeLU(h)] [Wo ; W2] (+ b_o + b2)
  s = make_map_2d(&tm_act, act, T, H + F, H + F, pb::kGemmBM);
  if (s != PB_OK) return s;
  EpiParams e2{};
  e2.bias = h->has_bias ? h->bias2 : nullptr;
  e2.resid = x;
  e2.y = y;
  PB_CUDA(pb::launch_gemm(pb::kEpiResidual, tm_act, h->tm_w2cat, T, H, H + F, e2, h->num_sms,
                          h->status, h->limit_ns, st),
          "second GEMM launch");
  return PB_OK;
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

pb_status run_stack(pb_handle* const* layers, int32_t n, const __nv_bfloat16* x,
                    __nv_bfloat16* y, uint8_t* scratch, cudaStream_t st) {
  const pb_scratch_layout L = scratch_layout(layers[0]->d);
  __nv_bfloat16* io[2] = {reinterpret_cast<__nv_bfloat16*>(scratch + L.io0),
                          reinterpret_cast<__nv_bfloat16*>(scratch + L.io1)};
  const __nv_bfloat16* in = x;
  int next = (in == io[0]) ? 1 : 0;
  for (int32_t l = 0; l < n; ++l) {
    __nv_bfloat16* out = (l == n - 1) ? y : io[next];
    pb_status s = run_block(layers[l], in, out, scratch, st);
    if (s != PB_OK) return s;
    in = out;
    next ^= 1;
  }
  return PB_OK;
}

}  // namespace

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
  pb_status s = check_dims(dims);
  if (s != PB_OK) return s;
  if (out == nullptr) return fail(PB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (w == nullptr) return fail(PB_ERR_INVALID_ARG, "weights is NULL");
  const void* req[6] = {w->ln_gamma, w->ln_beta, w->wqkv, w->w1, w->wo, w->w2};
  const char* names[6] = {"ln_gamma", "ln_beta", "wqkv", "w1", "wo", "w2"};
  for (int i = 0; i < 6; ++i) {
    if (req[i] == nullptr) return fail(PB_ERR_INVALID_ARG, "weights.%s is NULL", names[i]);
    if (!aligned(req[i], 16))
      return fail(PB_ERR_INVALID_ARG, "weights.%s is not 16-byte aligned", names[i]);
  }
  const void* opt[4] = {w->b_qkv, w->b1, w->b_o, w->b2};
  for (int i = 0; i < 4; ++i)
    if (opt[i] != nullptr && !aligned(opt[i], 2))
      return fail(PB_ERR_INVALID_ARG, "a bias pointer is misaligned");
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
  h->limit_ns = kDefaultLimitNs;
  h->ws = static_cast<uint8_t*>(workspace);
  h->status = reinterpret_cast<int*>(h->ws + L.status);
  h->w1cat = reinterpret_cast<__nv_bfloat16*>(h->ws + L.w1cat);
  h->w2cat = reinterpret_cast<__nv_bfloat16*>(h->ws + L.w2cat);
  h->bias1 = reinterpret_cast<float*>(h->ws + L.bias1);
  h->bias2 = reinterpret_cast<float*>(h->ws + L.bias2);
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
  // W1cat rows [0, 3H) = Wqkv^T, rows [3H, 3H + F) = W1^T
  PB_CUDA_H(pb::launch_transpose(bf(w->wqkv), H, 3 * H, 3 * H, h->w1cat, H, st), "pack Wqkv");
  PB_CUDA_H(pb::launch_transpose(bf(w->w1), H, F, F, h->w1cat + 3 * H * H, H, st), "pack W1");
  // W2cat columns [0, H) = Wo^T, columns [H, H + F) = W2^T
  PB_CUDA_H(pb::launch_transpose(bf(w->wo), H, H, H, h->w2cat, H + F, st), "pack Wo");
  PB_CUDA_H(pb::launch_transpose(bf(w->w2), F, H, H, h->w2cat + H, H + F, st), "pack W2");
  PB_CUDA_H(pb::launch_bias_prep(bf(w->b_qkv), bf(w->b1), bf(w->b_o), bf(w->b2), int(H), int(F),
                                 h->bias1, h->bias2, st),
            "bias prep");
  PB_CUDA_H(cudaMemcpyAsync(h->gamma, w->ln_gamma, H * 2, cudaMemcpyDeviceToDevice, st),
            "copy gamma");
  PB_CUDA_H(cudaMemcpyAsync(h->beta, w->ln_beta, H * 2, cudaMemcpyDeviceToDevice, st),
            "copy beta");
#undef PB_CUDA_H
  s = make_map_2d(&h->tm_w1cat, h->w1cat, 3 * H + F, H, H, pb::kGemmBN);
  if (s == PB_OK) s = make_map_2d(&h->tm_w2cat, h->w2cat, H, H + F, H + F, pb::kGemmBN);
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
  return run_block(h, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y),
                   static_cast<uint8_t*>(scratch), static_cast<cudaStream_t>(stream));
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
  return run_stack(layers, n_layers, static_cast<const __nv_bfloat16*>(x),
                   static_cast<__nv_bfloat16*>(y), static_cast<uint8_t*>(scratch),
                   static_cast<cudaStream_t>(stream));
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
  auto* io0 = reinterpret_cast<__nv_bfloat16*>(sc + L.io0);
  auto* io1 = reinterpret_cast<__nv_bfloat16*>(sc + L.io1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PB_CUDA(cudaMemcpyAsync(io0, x_host, n, cudaMemcpyHostToDevice, st), "copy x to the device");
  // The last layer writes into whichever io buffer did not hold its input.
  __nv_bfloat16* out = (n_layers % 2 == 1) ? io1 : io0;
  if (n_layers == 1) out = io1;
  s = run_stack(layers, n_layers, io0, out, sc, st);
  if (s != PB_OK) return s;
  PB_CUDA(cudaMemcpyAsync(y_host, out, n, cudaMemcpyDeviceToHost, st), "copy y to the host");
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

pb_status pb_destroy(pb_handle* h) {
  if (h == nullptr) return fail(PB_ERR_BAD_HANDLE, "handle is NULL");
  if (h->magic != kMagic) return fail(PB_ERR_BAD_HANDLE, "handle is destroyed or invalid");
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
  const void* ps[4] = {x, gamma, beta, out};
  for (const void* p : ps)
    if (p == nullptr || !aligned(p, 16))
      return fail(PB_ERR_INVALID_ARG, "pointers must be 16-byte aligned device pointers");
  PB_CUDA(pb::launch_layernorm(rows, H, static_cast<const __nv_bfloat16*>(x),
                               static_cast<const __nv_bfloat16*>(gamma),
                               static_cast<const __nv_bfloat16*>(beta), eps,
                               static_cast<__nv_bfloat16*>(out),
                               static_cast<cudaStream_t>(stream)),
          "layernorm launch");
  return PB_OK;
}

pb_status pb_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, const void* B, void* C,
                       int* status, void* stream) {
  if (M < 1 || N < 1 || K < 1) return fail(PB_ERR_INVALID_ARG, "M, N, K must be >= 1");
  if (K % 64 != 0 || N % 32 != 0)
    return fail(PB_ERR_UNSUPPORTED, "gemm needs K %% 64 == 0 and N %% 32 == 0");
  if (A == nullptr || B == nullptr || C == nullptr || !aligned(A, 16) || !aligned(B, 16) ||
      !aligned(C, 16))
    return fail(PB_ERR_INVALID_ARG, "A, B, C must be 16-byte aligned device pointers");
  int dev = -1, sms = 0;
  PB_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  PB_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
          "cudaDeviceGetAttribute");
  CUtensorMap ta, tb;
  pb_status s = make_map_2d(&ta, A, uint64_t(M), uint64_t(K), uint64_t(K), pb::kGemmBM);
  if (s == PB_OK) s = make_map_2d(&tb, B, uint64_t(N), uint64_t(K), uint64_t(K), pb::kGemmBN);
  if (s != PB_OK) return s;
  EpiParams ep{};
  ep.c = static_cast<__nv_bfloat16*>(C);
  ep.ldc = N;
  PB_CUDA(pb::launch_gemm(pb::kEpiStore, ta, tb, M, N, K, ep, sms, status, kDefaultLimitNs,
                          static_cast<cudaStream_t>(stream)),
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
  CUtensorMap tm_qk, tm_vt;
  const uint64_t dims3[3] = {uint64_t(2 * H), uint64_t(d.seq), uint64_t(d.batch)};
  const uint64_t str3[2] = {uint64_t(2 * H) * 2, uint64_t(2 * H) * 2 * uint64_t(d.seq)};
  const uint32_t box3[3] = {64, uint32_t(pb::kSwaBQ), 1};
  s = make_map(&tm_qk, qk, 3, dims3, str3, box3);
  if (s != PB_OK) return s;
  const uint64_t vdims[2] = {uint64_t(d.seq), uint64_t(d.batch) * uint64_t(H)};
  const uint64_t vstr[1] = {uint64_t(seq_pad) * 2};
  const uint32_t vbox[2] = {64, uint32_t(d.head_dim)};
  s = make_map(&tm_vt, vt, 2, vdims, vstr, vbox);
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
  sp.out = static_cast<__nv_bfloat16*>(act);
  sp.out_ld = act_ld;
  PB_CUDA(pb::launch_swa(tm_qk, tm_vt, sp, status, kDefaultLimitNs,
                         static_cast<cudaStream_t>(stream)),
          "attention launch");
  return PB_OK;
}

}  // extern "C"
