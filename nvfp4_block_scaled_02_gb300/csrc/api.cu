// api.cu -- the C ABI declared in include/nvfp4.h: argument validation (all
// synchronous, before anything is enqueued), output-buffer preparation on the
// caller's stream, and dispatch to the kernels.
#include <atomic>
#include <cstdint>

#include "launch.h"
#include "mx_quant.h"

namespace nvfp4 {

// SM count of the current device, looked up once per device (calls may come
// from several host threads: every thread stores the same value).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace nvfp4

namespace {

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Non-negative dimensions, each and their element count small enough for the
// byte offsets derived from them to fit in int64 (at most 8 bytes per
// element): a product that wrapped would size grids and checks from a wrong
// count.
constexpr int64_t kMaxElems = INT64_MAX >> 3;
bool dims_ok(int64_t s, int64_t r, int64_t c) {
  int64_t n = 0;
  return s >= 0 && r >= 0 && c >= 0 && s <= kMaxElems && r <= kMaxElems && c <= kMaxElems &&
         !__builtin_mul_overflow(r, c, &n) && !__builtin_mul_overflow(n, s, &n) &&
         n <= kMaxElems;
}

// 0 = 4/6 off, 1 = on with the MSE rule (compiled in), 2 = on, rule read at run time
int fos_mode(const nvfp4_config* cfg) {
  if (!cfg->four_over_six) return 0;
  return cfg->four_over_six_rule == NVFP4_FOS_MSE ? 1 : 2;
}

nvfp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

nvfp4_status check_out(const nvfp4_out* o, bool fos) {
  if (!o || !o->codes || !o->scales) return NVFP4_ERR_NULL;
  if (fos && !o->choice) return NVFP4_ERR_NULL;
  if (!aligned(o->codes, 16) || !aligned(o->scales, 16) || !aligned(o->dequant, 16))
    return NVFP4_ERR_ALIGN;
  if (fos && !aligned(o->choice, 16)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

// blocks == NVFP4_BLOCKS_TILE16: validation and dispatch.
nvfp4_status quantize_tile16(const nvfp4_config* cfg, const void* x, int64_t slices, int64_t rows,
                             int64_t cols, const float* global_amax, const nvfp4_out* row,
                             const nvfp4_out* col, int32_t* status, void* stream) {
  if (cfg->four_over_six) return NVFP4_ERR_ENUM;
  if (rows % 16 != 0 || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (slices == 0 || rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || !global_amax) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(global_amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  nvfp4_status e = check_out(row, false);
  if (e != NVFP4_OK) return e;
  if (col && (e = check_out(col, false)) != NVFP4_OK) return e;
  if (col && (row->dequant == nullptr) != (col->dequant == nullptr)) return NVFP4_ERR_NULL;
  nvfp4::Tile16Params p{};
  p.x = static_cast<const uint4*>(x);
  p.S = slices;
  p.R = rows;
  p.C = cols;
  p.gamax = global_amax;
  p.M = cfg->scale_max > 0.0f ? cfg->scale_max : 448.0f;
  p.seed = cfg->seed;
  p.step = cfg->step;
  p.r_codes = reinterpret_cast<uint32_t*>(row->codes);
  p.r_scales = row->scales;
  p.r_dq = static_cast<uint4*>(row->dequant);
  if (col) {
    p.c_codes = reinterpret_cast<uint32_t*>(col->codes);
    p.c_scales = col->scales;
    p.c_dq = static_cast<uint4*>(col->dequant);
  }
  p.status = status;
  return cuda_status(nvfp4::launch_quant_tile16(p, cfg->scale_fmt, cfg->rounding == NVFP4_ROUND_SR,
                                                static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_NULL: return "a required pointer is NULL";
    case NVFP4_ERR_SHAPE:
      return "invalid shape (negative, a size or element count above 2^60 - 1, or a blocked "
             "dimension not a multiple of 16)";
    case NVFP4_ERR_ALIGN: return "a pointer is not aligned as required";
    case NVFP4_ERR_ENUM: return "a configuration field is out of range";
    case NVFP4_ERR_CUDA: return "a CUDA launch failed";
  }
  return "unknown status";
}

nvfp4_status nvfp4_amax(const void* x, int64_t slices, int64_t rows, int64_t cols, float* amax,
                        int32_t* status, void* stream) {
  if (!dims_ok(slices, rows, cols)) return NVFP4_ERR_SHAPE;
  if (slices == 0) return NVFP4_OK;
  if (!amax) return NVFP4_ERR_NULL;
  if (rows * cols != 0 && !x) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  return cuda_status(nvfp4::launch_amax(static_cast<const uint16_t*>(x), slices, rows * cols, amax,
                                        status, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_amax_ws_bytes(int64_t slices) {
  return slices > 0 ? (size_t)slices * 2 * sizeof(uint32_t) : 0;
}

nvfp4_status nvfp4_amax_ws(const void* x, int64_t slices, int64_t rows, int64_t cols, float* amax,
                           void* workspace, size_t ws_bytes, int32_t* status, void* stream) {
  if (!dims_ok(slices, rows, cols)) return NVFP4_ERR_SHAPE;
  if (slices == 0) return NVFP4_OK;
  if (!amax || !workspace) return NVFP4_ERR_NULL;
  if (rows * cols != 0 && !x) return NVFP4_ERR_NULL;
  if (ws_bytes < nvfp4_amax_ws_bytes(slices)) return NVFP4_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(amax, 4) || !aligned(workspace, 4) || !aligned(status, 4))
    return NVFP4_ERR_ALIGN;
  return cuda_status(nvfp4::launch_amax_ticket(static_cast<const uint16_t*>(x), slices,
                                               rows * cols, amax,
                                               static_cast<uint32_t*>(workspace), status,
                                               static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_amax_noalloc(const void* x, int64_t slices, int64_t rows, int64_t cols,
                                float* amax, int32_t* status, void* stream) {
  if (!dims_ok(slices, rows, cols)) return NVFP4_ERR_SHAPE;
  if (slices > NVFP4_AMAX_NOALLOC_MAX_SLICES) return NVFP4_ERR_SHAPE;
  if (slices == 0) return NVFP4_OK;
  if (!amax) return NVFP4_ERR_NULL;
  if (rows * cols != 0 && !x) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  return cuda_status(nvfp4::launch_amax_noalloc(static_cast<const uint16_t*>(x), slices,
                                                rows * cols, amax, status,
                                                static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize(const nvfp4_config* cfg, const void* x, int64_t slices, int64_t rows,
                            int64_t cols, const float* global_amax, const nvfp4_out* row,
                            const nvfp4_out* col, int32_t* status, void* stream) {
  if (!cfg) return NVFP4_ERR_NULL;
  if (cfg->four_over_six_rule < 0 || cfg->four_over_six_rule > 2) return NVFP4_ERR_ENUM;
  if (cfg->blocks < 1 || cfg->blocks > 4 || cfg->scale_fmt < 0 || cfg->scale_fmt > 1 ||
      cfg->rounding < 0 || cfg->rounding > 1 || cfg->four_over_six < 0 || cfg->four_over_six > 1 ||
      !(cfg->scale_max >= 0.0f) || !(cfg->scale_max <= 3.402823466e+38f))
    return NVFP4_ERR_ENUM;
  if (!dims_ok(slices, rows, cols)) return NVFP4_ERR_SHAPE;
  if (cfg->blocks == NVFP4_BLOCKS_TILE16) return quantize_tile16(cfg, x, slices, rows, cols,
                                                                 global_amax, row, col, status,
                                                                 stream);
  const bool do_row = cfg->blocks & 1, do_col = cfg->blocks & 2;
  if (do_row && cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (do_col && rows % 16 != 0) return NVFP4_ERR_SHAPE;
  if (slices == 0 || rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || !global_amax) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(global_amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  const bool fos = cfg->four_over_six != 0, sr = cfg->rounding == NVFP4_ROUND_SR;
  if (do_row) {
    nvfp4_status e = check_out(row, fos);
    if (e != NVFP4_OK) return e;
  }
  if (do_col) {
    nvfp4_status e = check_out(col, fos);
    if (e != NVFP4_OK) return e;
  }
  const float M = cfg->scale_max > 0.0f ? cfg->scale_max : (fos ? 256.0f : 448.0f);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t Bs = rows * cols / 16, W = (Bs + 31) / 32;

  if (do_row && !do_col) {
    nvfp4::RowParams p{};
    p.x = static_cast<const uint4*>(x);
    p.Bs = Bs;
    p.W = W;
    p.gamax = global_amax;
    p.M = M;
    p.key = nvfp4::make_sr_key(cfg->seed, cfg->step);
    p.codes = reinterpret_cast<uint32_t*>(row->codes);
    p.scales = row->scales;
    p.choice = fos ? row->choice : nullptr;
    p.dq = static_cast<uint4*>(row->dequant);
    p.status = status;
    p.rule = cfg->four_over_six_rule;
    return cuda_status(nvfp4::launch_quant_row(p, slices, cfg->scale_fmt, sr, fos_mode(cfg), st));
  }
  // column blocks (alone or with row blocks): the bitmaps are OR-ed into
  if (fos) {
    const size_t bytes = (size_t)(slices * W) * sizeof(uint32_t);
    const int64_t words = (int64_t)(bytes / sizeof(uint32_t));
    if (do_row && nvfp4::launch_zero_words(row->choice, words, st) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    if (nvfp4::launch_zero_words(col->choice, words, st) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  nvfp4::DualParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.S = slices;
  p.R = rows;
  p.C = cols;
  p.gamax = global_amax;
  p.M = M;
  p.key = nvfp4::make_sr_key(cfg->seed, cfg->step);
  if (do_row) {
    p.r_codes = row->codes;
    p.r_scales = row->scales;
    p.r_choice = fos ? row->choice : nullptr;
    p.r_dq = static_cast<uint16_t*>(row->dequant);
  }
  p.c_codes = col->codes;
  p.c_scales = col->scales;
  p.c_choice = fos ? col->choice : nullptr;
  p.c_dq = static_cast<uint16_t*>(col->dequant);
  p.status = status;
  p.rule = cfg->four_over_six_rule;
  return cuda_status(
      nvfp4::launch_quant_dual(p, slices, do_row, cfg->scale_fmt, sr, fos_mode(cfg), st));
}

nvfp4_status nvfp4_quantize_per_token(const nvfp4_config* cfg, const void* x, int64_t rows,
                                      int64_t cols, float* row_amax, const nvfp4_out* out,
                                      int32_t* status, void* stream) {
  if (!cfg) return NVFP4_ERR_NULL;
  if (cfg->four_over_six_rule < 0 || cfg->four_over_six_rule > 2) return NVFP4_ERR_ENUM;
  if (cfg->blocks != NVFP4_BLOCKS_ROW || cfg->scale_fmt < 0 || cfg->scale_fmt > 1 ||
      cfg->rounding < 0 || cfg->rounding > 1 || cfg->four_over_six < 0 ||
      cfg->four_over_six > 1 || !(cfg->scale_max >= 0.0f) || !(cfg->scale_max <= 3.402823466e+38f))
    return NVFP4_ERR_ENUM;
  if (!dims_ok(1, rows, cols) || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || !row_amax) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(row_amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  const bool fos = cfg->four_over_six != 0;
  nvfp4_status e = check_out(out, fos);
  if (e != NVFP4_OK) return e;
  nvfp4::TokenParams p{};
  p.x = static_cast<const uint4*>(x);
  p.R = rows;
  p.C = cols;
  p.M = cfg->scale_max > 0.0f ? cfg->scale_max : (fos ? 256.0f : 448.0f);
  p.key = nvfp4::make_sr_key(cfg->seed, cfg->step);
  p.row_amax = row_amax;
  p.codes = reinterpret_cast<uint32_t*>(out->codes);
  p.scales = out->scales;
  p.choice = fos ? out->choice : nullptr;
  p.dq = static_cast<uint4*>(out->dequant);
  p.status = status;
  p.rule = cfg->four_over_six_rule;
  return cuda_status(nvfp4::launch_quant_token(p, cfg->scale_fmt, cfg->rounding == NVFP4_ROUND_SR,
                                               fos_mode(cfg), static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_requant_transpose(const nvfp4_config* src, const nvfp4_config* dst,
                                     int32_t target, const uint8_t* codes, const uint8_t* scales,
                                     int64_t slices, int64_t rows, int64_t cols,
                                     const float* global_amax, const nvfp4_out* out,
                                     int32_t* status, void* stream) {
  if (!src || !dst) return NVFP4_ERR_NULL;
  if (target < 0 || target > 1) return NVFP4_ERR_ENUM;
  if (src->scale_fmt < 0 || src->scale_fmt > 1 || src->four_over_six < 0 ||
      src->four_over_six > 1 || !(src->scale_max >= 0.0f) ||
      !(src->scale_max <= 3.402823466e+38f))
    return NVFP4_ERR_ENUM;
  if (dst->rounding < 0 || dst->rounding > 1) return NVFP4_ERR_ENUM;
  const bool nv = target == NVFP4_TARGET_NVFP4;
  if (nv && (dst->scale_fmt < 0 || dst->scale_fmt > 1 || dst->four_over_six < 0 ||
             dst->four_over_six > 1 || dst->four_over_six_rule < 0 ||
             dst->four_over_six_rule > 2 || !(dst->scale_max >= 0.0f) ||
             !(dst->scale_max <= 3.402823466e+38f)))
    return NVFP4_ERR_ENUM;
  if (!dims_ok(slices, rows, cols) || cols % 16 != 0 || rows % (nv ? 16 : 32) != 0)
    return NVFP4_ERR_SHAPE;
  if (slices == 0 || rows == 0 || cols == 0) return NVFP4_OK;
  if (!codes || !scales || !global_amax || !out || !out->codes || !out->scales)
    return NVFP4_ERR_NULL;
  const bool fos = nv && dst->four_over_six != 0;
  if (fos && !out->choice) return NVFP4_ERR_NULL;
  if (out->dequant) return NVFP4_ERR_ENUM;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(global_amax, 4) ||
      !aligned(status, 4) || !aligned(out->codes, 16) || !aligned(out->scales, 16) ||
      (fos && !aligned(out->choice, 16)))
    return NVFP4_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (fos) {
    const size_t W = (size_t)((rows * cols / 16 + 31) / 32);
    if (nvfp4::launch_zero_words(out->choice, (int64_t)(slices * W), st) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  nvfp4::RequantParams p{};
  p.codes = codes;
  p.scales = scales;
  p.S = slices;
  p.R = rows;
  p.C = cols;
  p.gamax = global_amax;
  p.src_fmt = src->scale_fmt;
  p.M_src = src->scale_max > 0.0f ? src->scale_max : (src->four_over_six ? 256.0f : 448.0f);
  p.M_dst = dst->scale_max > 0.0f ? dst->scale_max : (fos ? 256.0f : 448.0f);
  p.key = nvfp4::make_sr_key(dst->seed, dst->step);
  p.out_codes = out->codes;
  p.out_scales = out->scales;
  p.out_choice = fos ? out->choice : nullptr;
  p.status = status;
  p.rule = dst->four_over_six_rule;
  return cuda_status(nvfp4::launch_requant(p, target, dst->scale_fmt, dst->rounding == NVFP4_ROUND_SR,
                                           nv ? fos_mode(dst) : 0, st));
}

nvfp4_status nvfp4_mx_quantize(const nvfp4_config* cfg, const void* x, int64_t slices,
                               int64_t rows, int64_t cols, const nvfp4_out* row,
                               const nvfp4_out* col, int32_t* status, void* stream) {
  if (!cfg) return NVFP4_ERR_NULL;
  if (cfg->blocks < 1 || cfg->blocks > 3 || cfg->rounding < 0 || cfg->rounding > 1)
    return NVFP4_ERR_ENUM;
  const bool do_row = cfg->blocks & 1, do_col = cfg->blocks & 2;
  if (!dims_ok(slices, rows, cols) || (do_row && cols % 32 != 0) ||
      (do_col && rows % 32 != 0))
    return NVFP4_ERR_SHAPE;
  if (slices == 0 || rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || (do_row && (!row || !row->codes || !row->scales)) ||
      (do_col && (!col || !col->codes || !col->scales)))
    return NVFP4_ERR_NULL;
  if ((do_row && row->dequant) || (do_col && col->dequant)) return NVFP4_ERR_ENUM;
  if (!aligned(x, 16) || !aligned(status, 4) ||
      (do_row && (!aligned(row->codes, 16) || !aligned(row->scales, 16))) ||
      (do_col && (!aligned(col->codes, 16) || !aligned(col->scales, 16))))
    return NVFP4_ERR_ALIGN;
  nvfp4::MxParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.S = slices;
  p.R = rows;
  p.C = cols;
  p.seed = cfg->seed;
  p.step = cfg->step;
  if (do_row) {
    p.r_codes = row->codes;
    p.r_scales = row->scales;
  }
  if (do_col) {
    p.c_codes = col->codes;
    p.c_scales = col->scales;
  }
  p.status = status;
  return cuda_status(nvfp4::launch_mx_quant(p, do_row, do_col, cfg->rounding == NVFP4_ROUND_SR,
                                            static_cast<cudaStream_t>(stream)));
}

static nvfp4_status ste_common(const void* x, int64_t rows, int64_t cols, const float* s_pre) {
  if (!dims_ok(1, rows, cols) || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || !s_pre) return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(s_pre, 4)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

nvfp4_status nvfp4_fakequant_fwd(const void* x, int64_t rows, int64_t cols, const float* s_pre,
                                 const float* s_post, void* xq, int32_t* status, void* stream) {
  nvfp4_status e = ste_common(x, rows, cols, s_pre);
  if (e != NVFP4_OK || rows == 0 || cols == 0) return e;
  if (!xq) return NVFP4_ERR_NULL;
  if (!aligned(xq, 16) || !aligned(s_post, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  nvfp4::SteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.nblocks = rows * cols / 16;
  p.s_pre = s_pre;
  p.s_post = s_post;
  p.out = static_cast<uint4*>(xq);
  p.status = status;
  return cuda_status(nvfp4::launch_fakequant_fwd(p, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_scale_grad_bwd(const void* x, const void* gq, int64_t rows, int64_t cols,
                                  const float* s_pre, const float* s_post, void* gx,
                                  float* gs_pre, float* gs_post, int32_t* status, void* stream) {
  nvfp4_status e = ste_common(x, rows, cols, s_pre);
  if (e != NVFP4_OK || rows == 0 || cols == 0) return e;
  if (!gq || !gs_pre) return NVFP4_ERR_NULL;
  if (s_post && !gs_post) return NVFP4_ERR_NULL;
  if (!s_post && gs_post) return NVFP4_ERR_NULL;
  if (!aligned(gq, 16) || !aligned(gx, 16) || !aligned(gs_pre, 4) || !aligned(gs_post, 4) ||
      !aligned(s_post, 4) || !aligned(status, 4))
    return NVFP4_ERR_ALIGN;
  nvfp4::SteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.gq = static_cast<const uint4*>(gq);
  p.nblocks = rows * cols / 16;
  p.s_pre = s_pre;
  p.s_post = s_post;
  p.out = static_cast<uint4*>(gx);
  p.gs_pre = gs_pre;
  p.gs_post = gs_post;
  p.status = status;
  return cuda_status(nvfp4::launch_scale_grad_bwd(p, static_cast<cudaStream_t>(stream)));
}

static nvfp4_status fp8_common(const float* global_amax, int32_t* status) {
  if (!global_amax) return NVFP4_ERR_NULL;
  if (!aligned(global_amax, 4) || !aligned(status, 4)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

nvfp4_status nvfp4_fakequant_fwd_fp8scale(const void* x, int64_t rows, int64_t cols,
                                          const float* s_pre, const float* s_post,
                                          const float* global_amax, void* xq, int32_t* status,
                                          void* stream) {
  nvfp4_status e = ste_common(x, rows, cols, s_pre);
  if (e != NVFP4_OK || rows == 0 || cols == 0) return e;
  if ((e = fp8_common(global_amax, status)) != NVFP4_OK) return e;
  if (!xq) return NVFP4_ERR_NULL;
  if (!aligned(xq, 16) || !aligned(s_post, 4)) return NVFP4_ERR_ALIGN;
  nvfp4::SteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.nblocks = rows * cols / 16;
  p.s_pre = s_pre;
  p.s_post = s_post;
  p.out = static_cast<uint4*>(xq);
  p.status = status;
  p.gamax = global_amax;
  return cuda_status(nvfp4::launch_fakequant_fwd(p, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_scale_grad_bwd_fp8scale(const void* x, const void* gq, int64_t rows,
                                           int64_t cols, const float* s_pre, const float* s_post,
                                           const float* global_amax, void* gx, float* gs_pre,
                                           float* gs_post, int32_t* status, void* stream) {
  nvfp4_status e = ste_common(x, rows, cols, s_pre);
  if (e != NVFP4_OK || rows == 0 || cols == 0) return e;
  if ((e = fp8_common(global_amax, status)) != NVFP4_OK) return e;
  if (!gq || !gs_pre) return NVFP4_ERR_NULL;
  if (s_post && !gs_post) return NVFP4_ERR_NULL;
  if (!s_post && gs_post) return NVFP4_ERR_NULL;
  if (!aligned(gq, 16) || !aligned(gx, 16) || !aligned(gs_pre, 4) || !aligned(gs_post, 4) ||
      !aligned(s_post, 4))
    return NVFP4_ERR_ALIGN;
  nvfp4::SteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.gq = static_cast<const uint4*>(gq);
  p.nblocks = rows * cols / 16;
  p.s_pre = s_pre;
  p.s_post = s_post;
  p.out = static_cast<uint4*>(gx);
  p.gs_pre = gs_pre;
  p.gs_post = gs_post;
  p.status = status;
  p.gamax = global_amax;
  return cuda_status(nvfp4::launch_scale_grad_bwd(p, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_scale_init_mse(const void* x, int64_t rows, int64_t cols,
                                  const float* global_amax, uint8_t* scale_codes, float* s,
                                  int32_t* status, void* stream) {
  if (!dims_ok(1, rows, cols) || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return NVFP4_OK;
  if (!x || (!scale_codes && !s)) return NVFP4_ERR_NULL;
  nvfp4_status e = fp8_common(global_amax, status);
  if (e != NVFP4_OK) return e;
  if (!aligned(x, 16) || !aligned(s, 4)) return NVFP4_ERR_ALIGN;
  nvfp4::ScaleInitParams p{};
  p.x = static_cast<const uint4*>(x);
  p.nblocks = rows * cols / 16;
  p.gamax = global_amax;
  p.codes = scale_codes;
  p.s = s;
  p.status = status;
  return cuda_status(nvfp4::launch_scale_init_mse(p, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_export_scales(const void* x, int64_t rows, int64_t cols, const float* s_pre,
                                 const float* s_post, const float* global_amax,
                                 const nvfp4_out* out, int32_t* status, void* stream) {
  nvfp4_status e = ste_common(x, rows, cols, s_pre);
  if (e != NVFP4_OK || rows == 0 || cols == 0) return e;
  if ((e = fp8_common(global_amax, status)) != NVFP4_OK) return e;
  if (!out || !out->codes || !out->scales) return NVFP4_ERR_NULL;
  if (out->dequant) return NVFP4_ERR_ENUM;
  if (!aligned(out->codes, 16) || !aligned(out->scales, 16) || !aligned(s_post, 4))
    return NVFP4_ERR_ALIGN;
  nvfp4::SteParams p{};
  p.x = static_cast<const uint4*>(x);
  p.nblocks = rows * cols / 16;
  p.s_pre = s_pre;
  p.s_post = s_post;
  p.status = status;
  p.gamax = global_amax;
  p.codes = out->codes;
  p.scales = out->scales;
  return cuda_status(nvfp4::launch_export_scales(p, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_codec_probe(int32_t op, const float* in, const uint32_t* aux, int64_t n,
                               uint8_t* out, void* stream) {
  if (op < 0 || op > 7) return NVFP4_ERR_ENUM;
  if (n < 0 || n > kMaxElems) return NVFP4_ERR_SHAPE;
  if (n == 0) return NVFP4_OK;
  if (!in || !out || ((op == 3 || op == 5 || op == 7) && !aux)) return NVFP4_ERR_NULL;
  if (!aligned(in, 4) || !aligned(aux, 4)) return NVFP4_ERR_ALIGN;
  return cuda_status(
      nvfp4::launch_codec_probe(op, in, aux, n, out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_sr_bits(uint32_t seed, uint32_t step, uint32_t direction, uint64_t idx0,
                           int64_t n, uint32_t* out, void* stream) {
  if (n < 0 || n > kMaxElems) return NVFP4_ERR_SHAPE;
  if (n == 0) return NVFP4_OK;
  if (!out) return NVFP4_ERR_NULL;
  if (!aligned(out, 4)) return NVFP4_ERR_ALIGN;
  return cuda_status(nvfp4::launch_sr_bits(seed, step, direction, idx0, n, out,
                                           static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
