// C ABI of libmla: argument checks, workspace planning and kernel dispatch.
// Every entry point checks its arguments before it queues anything. None of
// them allocates device memory except mla_absorb_weights.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "mla_internal.h"

// Per-device error word. Kernels OR MLA_DEVERR_* bits into it.
__device__ uint32_t g_mla_device_error = 0;

namespace mla {

namespace {

constexpr int kMaxDevices = 64;

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

struct DeviceInfo {
  bool ready = false;
  int sms = 0, major = 0, minor = 0;
  int tc_pairs = 0;  // CTA pairs the tensor-core attention grid holds (0: unavailable)
  uint32_t* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Queries (once per device) the SM count, compute capability and the device
// address of the error word. Must run with the device current.
const DeviceInfo* device_info() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[d];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err), g_mla_device_error) !=
            cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (di.major == 10 && di.minor == 3) di.tc_pairs = attend_tc_max_pairs();
    di.ready = true;
  }
  return &di;
}

mla_status check_config(const mla_config* c) {
  if (!c) return MLA_ERR_INVALID_ARG;
  if (c->dtype != MLA_F32 && c->dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (c->impl < MLA_IMPL_AUTO || c->impl > MLA_IMPL_TENSOR_CORE) return MLA_ERR_INVALID_ARG;
  if (!(c->rope_base > 0.f) || !std::isfinite(c->rope_base)) return MLA_ERR_INVALID_ARG;
  if (!(c->softmax_scale >= 0.f) || !std::isfinite(c->softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (c->n_h < 1 || c->d_model < 1 || c->d_nope < 1 || c->d_v < 1 || c->block_size < 1)
    return MLA_ERR_SHAPE;
  if (c->d_c < 4 || c->d_c > 512 || c->d_c % 4 != 0) return MLA_ERR_SHAPE;
  if (c->d_r < 2 || c->d_r % 2 != 0 || c->d_c + c->d_r > 1024) return MLA_ERR_SHAPE;
  // d_v: the CUDA-core combine keeps [2][16][d_v] fp32 partial outputs in
  // shared memory beside o_lat and the merge weights (about 191 KB at
  // d_c = 512, d_v = 1024 on 148 SMs, under the 227 KB a block may use).
  if (c->d_nope > 1024 || c->d_v > 1024) return MLA_ERR_SHAPE;
  return MLA_OK;
}

Shape shape_of(const mla_config* c) {
  Shape s;
  s.n_h = c->n_h;
  s.d_model = c->d_model;
  s.d_c = c->d_c;
  s.d_r = c->d_r;
  s.d_nope = c->d_nope;
  s.d_v = c->d_v;
  s.bs = c->block_size;
  s.rope_base = c->rope_base;
  s.scale = c->softmax_scale > 0.f ? c->softmax_scale
                                   : 1.0f / std::sqrt(static_cast<float>(c->d_nope + c->d_r));
  return s;
}

int dtype_bytes(mla_dtype d) { return d == MLA_F32 ? 4 : 2; }

bool tc_device(const DeviceInfo* di) {
  return di && di->major == 10 && di->minor == 3 && di->tc_pairs > 0;
}

// Decode kernel for this config on this device, or -1 if the requested one cannot run.
int resolve_impl(const mla_config* c, const DeviceInfo* di) {
  const Shape s = shape_of(c);
  const bool tc_ok = attend_tc_supported(s, c->dtype) && tc_device(di);
  if (c->impl == MLA_IMPL_TENSOR_CORE) return tc_ok ? MLA_IMPL_TENSOR_CORE : -1;
  if (c->impl == MLA_IMPL_CUDA_CORE) return MLA_IMPL_CUDA_CORE;
  return tc_ok ? MLA_IMPL_TENSOR_CORE : MLA_IMPL_CUDA_CORE;
}

mla_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  cudaGetLastError();
  return MLA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

struct Plan {
  Shape s;
  int impl;
  Partition part;
  WsLayout lay;
};

mla_status make_plan(const mla_config* cfg, int B, int n_q, const DeviceInfo* di, int impl,
                     Plan* out) {
  out->s = shape_of(cfg);
  out->impl = impl;
  out->part = partition_for(impl, out->s, B, n_q, di->sms, di->tc_pairs);
  out->lay = ws_layout(out->s, impl == MLA_IMPL_CUDA_CORE ? 4 : dtype_bytes(cfg->dtype), B, n_q,
                       out->part);
  return MLA_OK;
}

mla_status check_decode_args(const mla_config* cfg, int B, int n_q) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (B < 1 || n_q < 1) return MLA_ERR_SHAPE;
  const long long rows = static_cast<long long>(B) * n_q * cfg->n_h;
  if (rows > (1LL << 30)) return MLA_ERR_SHAPE;
  return MLA_OK;
}

}  // namespace

Partition partition_for(int impl, const Shape& s, int B, int n_q, int num_sms, int tc_pairs) {
  Partition p;
  const int rows = n_q * s.n_h;
  if (impl == MLA_IMPL_TENSOR_CORE) {
    // 128 query rows per group (the MMA's M); one work range per CTA pair
    p.RG = 128;
    p.TS = 64;
    p.C = tc_pairs;
    p.K = 4;  // a piece change stalls the pair's pipeline for about 4 tiles
  } else {
    p.RG = 16;
    p.TS = 64;
    p.C = num_sms * 3;
    p.K = 0;
  }
  p.G = (rows + p.RG - 1) / p.RG;
  p.slots = p.C + p.G * B;
  return p;
}

WsLayout ws_layout(const Shape& s, int q_bytes, int B, int n_q, const Partition& p) {
  WsLayout l;
  size_t off = 0;
  l.qabs = off;
  off = align256(off + static_cast<size_t>(B) * n_q * s.n_h * s.R() * q_bytes);
  l.tiles = off;
  off = align256(off + sizeof(int32_t) * B);
  l.prefix = off;
  off = align256(off + sizeof(int32_t) * (B + 1));
  l.bounds = off;
  off = align256(off + sizeof(long long) * (p.C + 1));
  l.first_b = off;
  off = align256(off + sizeof(int32_t) * p.C);
  l.part_o = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(p.slots) * p.RG * s.d_c);
  l.part_lse = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(p.slots) * p.RG);
  l.total = off;
  return l;
}

WsView ws_view(void* base, const WsLayout& l) {
  char* b = static_cast<char*>(base);
  WsView v;
  v.qabs = b + l.qabs;
  v.tiles = reinterpret_cast<int32_t*>(b + l.tiles);
  v.prefix = reinterpret_cast<int32_t*>(b + l.prefix);
  v.bounds = reinterpret_cast<long long*>(b + l.bounds);
  v.first_b = reinterpret_cast<int32_t*>(b + l.first_b);
  v.part_o = reinterpret_cast<float*>(b + l.part_o);
  v.part_lse = reinterpret_cast<float*>(b + l.part_lse);
  return v;
}

}  // namespace mla

struct mla_weights_s {
  mla::Weights w;
  mla_config cfg;
};

struct mla_full_weights_s {
  mla::FullWeights w;
  mla_config cfg;
};

using namespace mla;

namespace {

// RoPE frequencies theta_i = base^(-2i/d_r), stored for the device as
// theta_i / (2 pi) in units of 2^-64 turns (round to nearest). Extended
// precision on the host keeps the stored fraction within half a unit.
void rope_turn_table(float base, int d_r, uint64_t* out) {
  const long double two_pi = 8.0L * std::atan(1.0L);
  for (int i = 0; i < d_r / 2; ++i) {
    const long double theta = std::pow(static_cast<long double>(base), -2.0L * i / d_r);
    out[i] = static_cast<uint64_t>(std::ldexp(theta / two_pi, 64) + 0.5L);
  }
}

bool same_shape(const mla_config* a, const mla_config* b) {
  return a->n_h == b->n_h && a->d_model == b->d_model && a->d_c == b->d_c && a->d_r == b->d_r &&
         a->d_nope == b->d_nope && a->d_v == b->d_v && a->dtype == b->dtype;
}

// Resolves the decode kernel and checks the workspace for one decode call.
// Only the fused mla_decode may move from the tensor-core kernel to the
// CUDA-core one for a misaligned cache: the stage calls must agree on one
// partition, so they reject such a cache instead.
mla_status prepare_decode(const mla_config* cfg, int B, int n_q, const void* cache,
                          const void* workspace, size_t ws_bytes, Plan* plan,
                          const DeviceInfo** di_out, bool allow_fallback = false) {
  mla_status st = check_decode_args(cfg, B, n_q);
  if (st != MLA_OK) return st;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  int impl = resolve_impl(cfg, di);
  if (impl < 0) return MLA_ERR_UNSUPPORTED;
  if (impl == MLA_IMPL_TENSOR_CORE && cache && !aligned16(cache)) {
    if (!allow_fallback || cfg->impl == MLA_IMPL_TENSOR_CORE) return MLA_ERR_INVALID_ARG;
    impl = MLA_IMPL_CUDA_CORE;
  }
  make_plan(cfg, B, n_q, di, impl, plan);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MLA_ERR_WORKSPACE;
  if (ws_bytes < plan->lay.total) return MLA_ERR_WORKSPACE;
  *di_out = di;
  return MLA_OK;
}

// The fp8 cache runs on the tensor-core kernels only: bf16 weights and
// queries at the DeepSeek-V2 latent widths, 64-token blocks, a B300.
bool fp8_supported(const mla_config* cfg, const DeviceInfo* di) {
  const Shape s = shape_of(cfg);
  return cfg->dtype == MLA_BF16 && cfg->impl != MLA_IMPL_CUDA_CORE && s.d_nope == 128 &&
         s.d_v == 128 && attend_tc_supported(s, cfg->dtype) &&
         absorb_tc_supported(s, cfg->dtype) && combine_tc_supported(s, cfg->dtype) &&
         tc_device(di);
}

constexpr int kFp8AppendChunk = 256;  // tokens whose fp32 rows the workspace holds

// Device scratch of mla_decode_full beyond the per-head decode's workspace:
// the fp32 query projection [B*n_q][n_h*R] (reused for o_lat, which is no
// wider), then the split partials of the two x W products.
struct FullExtra {
  XwPlan q, o;
  size_t proj, part, total;
};

FullExtra full_extra(const Shape& s, int B, int n_q, int sms) {
  FullExtra f;
  const int M = B * n_q;
  f.q = xw_plan(M, s.d_model, s.n_h * s.R(), sms);
  f.o = xw_plan(M, s.n_h * s.d_c, s.d_model, sms);
  f.proj = align256(sizeof(float) * static_cast<size_t>(M) * s.n_h * s.R());
  const size_t pq = xw_part_floats(M, s.n_h * s.R(), f.q);
  const size_t po = xw_part_floats(M, s.d_model, f.o);
  f.part = align256(sizeof(float) * (pq > po ? pq : po));
  f.total = f.proj + f.part;
  return f;
}

}  // namespace

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE";
    case MLA_ERR_CAPACITY: return "MLA_ERR_CAPACITY";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_CHECK: return "MLA_ERR_DEVICE_CHECK";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
  }
  return "MLA_ERR_UNKNOWN";
}

mla_status mla_absorb_weights(const mla_config* cfg, const void* W_dkv, const void* W_kr,
                              const void* W_uk, const void* W_uv, cudaStream_t stream,
                              mla_weights* out) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!W_dkv || !W_kr || !W_uk || !W_uv) return MLA_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return MLA_ERR_CUDA;
  const Shape s = shape_of(cfg);
  const size_t eb = dtype_bytes(cfg->dtype);
  mla_weights_s* h = new (std::nothrow) mla_weights_s();
  if (!h) return MLA_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->w.shape = s;
  h->w.dtype = cfg->dtype;
  h->w.device = dev;
  const size_t n_dkvr = static_cast<size_t>(s.R()) * s.d_model * eb;
  const size_t n_uk = static_cast<size_t>(s.n_h) * s.d_c * s.d_nope * eb;
  const size_t n_uv = static_cast<size_t>(s.n_h) * s.d_c * s.d_v * eb;
  const int half = s.d_r / 2;
  auto release = [h]() {
    cudaFree(h->w.w_dkvr);
    cudaFree(h->w.w_uk);
    cudaFree(h->w.w_uv);
    cudaFree(h->w.rope_turns);
    delete h;
  };
  if (cudaMalloc(&h->w.w_dkvr, n_dkvr) != cudaSuccess ||
      cudaMalloc(&h->w.w_uk, n_uk) != cudaSuccess || cudaMalloc(&h->w.w_uv, n_uv) != cudaSuccess ||
      cudaMalloc(&h->w.rope_turns, sizeof(uint64_t) * half) != cudaSuccess) {
    cudaGetLastError();
    release();
    return MLA_ERR_CUDA;
  }
  uint64_t turns[512];
  rope_turn_table(cfg->rope_base, s.d_r, turns);
  cudaError_t e = cudaMemcpyAsync(h->w.rope_turns, turns, sizeof(uint64_t) * half,
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess)
    e = launch_pack_weights(s, cfg->dtype, W_dkv, W_kr, W_uk, W_uv, &h->w, stream);
  // The decode kernels load the packed weights before they wait for their
  // predecessor on the stream, so the packing has to be complete here.
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaStreamSynchronize(stream);
    release();
    return MLA_ERR_CUDA;
  }
  *out = h;
  return MLA_OK;
}

mla_status mla_weights_free(mla_weights w) {
  if (!w) return MLA_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(w->w.device);
  cudaDeviceSynchronize();
  cudaFree(w->w.w_dkvr);
  cudaFree(w->w.w_uk);
  cudaFree(w->w.w_uv);
  cudaFree(w->w.rope_turns);
  if (prev >= 0) cudaSetDevice(prev);
  delete w;
  return MLA_OK;
}

mla_status mla_append_kv(const mla_config* cfg, mla_weights w, const void* x,
                         const int32_t* seq_idx, const int32_t* pos, const int32_t* page_table,
                         int32_t B, int32_t max_blocks, void* cache, int32_t num_blocks,
                         int32_t T, cudaStream_t stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!w) return MLA_ERR_INVALID_ARG;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (T < 0 || B < 1 || max_blocks < 1 || num_blocks < 1) return MLA_ERR_SHAPE;
  if (T == 0) return MLA_OK;
  if (!x || !seq_idx || !pos || !page_table || !cache) return MLA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  return from_cuda(launch_append(shape_of(cfg), cfg->dtype, &w->w, x, seq_idx, pos, page_table, B,
                                 max_blocks, cache, num_blocks, T, di->err, stream));
}

mla_status mla_decode_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                     int64_t total_tokens, size_t* bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = 0;
  mla_status st = check_decode_args(cfg, B, n_q);
  if (st != MLA_OK) return st;
  if (total_tokens < 0) return MLA_ERR_SHAPE;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  const int impl = resolve_impl(cfg, di);
  if (impl < 0) return MLA_ERR_UNSUPPORTED;
  Plan p;
  make_plan(cfg, B, n_q, di, impl, &p);
  size_t need = p.lay.total;
  if (cfg->impl == MLA_IMPL_AUTO && impl == MLA_IMPL_TENSOR_CORE) {
    // a misaligned cache falls back to the CUDA-core kernel: cover that too
    Plan q;
    make_plan(cfg, B, n_q, di, MLA_IMPL_CUDA_CORE, &q);
    if (q.lay.total > need) need = q.lay.total;
  }
  *bytes = need;
  return MLA_OK;
}

mla_status mla_decode_impl(const mla_config* cfg, int32_t* impl) {
  if (!impl) return MLA_ERR_INVALID_ARG;
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  const int r = resolve_impl(cfg, di);
  if (r < 0) return MLA_ERR_UNSUPPORTED;
  *impl = r;
  return MLA_OK;
}

mla_status mla_decode_absorb_q(const mla_config* cfg, mla_weights w, const void* q,
                               const int32_t* seq_lens, int32_t max_blocks, int32_t B,
                               int32_t n_q, void* workspace, size_t ws_bytes,
                               cudaStream_t stream) {
  if (!w || !q || !seq_lens) return MLA_ERR_INVALID_ARG;
  if (max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, nullptr, workspace, ws_bytes, &p, &di);
  if (st != MLA_OK) return st;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  const WsView v = ws_view(workspace, p.lay);
  // The tensor-core attention reads queries pre-multiplied by scale * log2(e).
  const float out_scale =
      p.impl == MLA_IMPL_TENSOR_CORE ? p.s.scale * 1.4426950408889634f : 1.f;
  if (p.impl == MLA_IMPL_TENSOR_CORE && absorb_tc_supported(p.s, cfg->dtype) && aligned16(q))
    return from_cuda(launch_absorb_q_tc(p.s, &w->w, q, seq_lens, max_blocks, B, n_q, p.part, v,
                                        out_scale, false, di->err, stream));
  return from_cuda(launch_absorb_q(p.s, cfg->dtype, &w->w, q, seq_lens, max_blocks, B, n_q,
                                   p.part, v, out_scale, p.impl == MLA_IMPL_CUDA_CORE, di->err,
                                   stream));
}

mla_status mla_decode_attend(const mla_config* cfg, const void* cache, int32_t num_blocks,
                             const int32_t* page_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t n_q, void* workspace,
                             size_t ws_bytes, cudaStream_t stream) {
  if (!cache || !page_table || !seq_lens) return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, cache, workspace, ws_bytes, &p, &di);
  if (st != MLA_OK) return st;
  if (static_cast<long long>(num_blocks) * cfg->block_size > (1LL << 31) - 1) return MLA_ERR_SHAPE;
  const WsView v = ws_view(workspace, p.lay);
  cudaError_t e;
  if (p.impl == MLA_IMPL_TENSOR_CORE)
    e = launch_attend_tc(p.s, cache, num_blocks, page_table, max_blocks, B, n_q, p.part, v,
                         seq_lens, di->err, stream);
  else
    e = launch_attend_simt(p.s, cfg->dtype, cache, num_blocks, page_table, max_blocks, B, n_q,
                           p.part, v, seq_lens, di->err, stream);
  return from_cuda(e);
}

mla_status mla_decode_combine(const mla_config* cfg, mla_weights w, const int32_t* seq_lens,
                              int32_t B, int32_t n_q, float* out, void* workspace,
                              size_t ws_bytes, cudaStream_t stream) {
  if (!w || !out || !seq_lens) return MLA_ERR_INVALID_ARG;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, nullptr, workspace, ws_bytes, &p, &di);
  if (st != MLA_OK) return st;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  const WsView v = ws_view(workspace, p.lay);
  // (the tensor-core combine writes out in 16-byte vectors)
  if (p.impl == MLA_IMPL_TENSOR_CORE && combine_tc_supported(p.s, cfg->dtype) && aligned16(out))
    return from_cuda(launch_combine_tc(p.s, &w->w, B, n_q, p.part, v, out, nullptr, di->err, stream));
  return from_cuda(launch_combine(p.s, cfg->dtype, &w->w, seq_lens, B, n_q, p.part, v, out,
                                  stream));
}

mla_status mla_decode(const mla_config* cfg, mla_weights w, const void* q, const void* cache,
                      int32_t num_blocks, const int32_t* page_table, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t B, int32_t n_q, float* out,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!w || !q || !cache || !page_table || !seq_lens || !out) return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, cache, workspace, ws_bytes, &p, &di, true);
  if (st != MLA_OK) return st;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * cfg->block_size > (1LL << 31) - 1) return MLA_ERR_SHAPE;
  // The three stages below see the same config, so they resolve the same
  // kernel and partition as this call did.
  mla_config c2 = *cfg;
  c2.impl = p.impl;
  st = mla_decode_absorb_q(&c2, w, q, seq_lens, max_blocks, B, n_q, workspace, ws_bytes, stream);
  if (st != MLA_OK) return st;
  st = mla_decode_attend(&c2, cache, num_blocks, page_table, max_blocks, seq_lens, B, n_q,
                         workspace, ws_bytes, stream);
  if (st != MLA_OK) return st;
  return mla_decode_combine(&c2, w, seq_lens, B, n_q, out, workspace, ws_bytes, stream);
}

mla_status mla_decode_latent(const mla_config* cfg, const void* q_abs, const void* cache,
                             int32_t num_blocks, const int32_t* page_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t n_q, float* o_lat,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!q_abs || !cache || !page_table || !seq_lens || !o_lat) return MLA_ERR_INVALID_ARG;
  // both merge kernels write o_lat in 16-byte vectors
  if (!aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, cache, workspace, ws_bytes, &p, &di, true);
  if (st != MLA_OK) return st;
  if (static_cast<long long>(num_blocks) * cfg->block_size > (1LL << 31) - 1) return MLA_ERR_SHAPE;
  const WsView v = ws_view(workspace, p.lay);
  const bool tc = p.impl == MLA_IMPL_TENSOR_CORE;
  // the tensor-core attention reads queries pre-multiplied by scale * log2(e)
  const float out_scale = tc ? p.s.scale * 1.4426950408889634f : 1.f;
  cudaError_t e = launch_latent_q(p.s, cfg->dtype, q_abs, seq_lens, max_blocks, B, n_q, p.part, v,
                                  out_scale, !tc, di->err, stream);
  if (e == cudaSuccess) {
    if (tc)
      e = launch_attend_tc(p.s, cache, num_blocks, page_table, max_blocks, B, n_q, p.part, v,
                           seq_lens, di->err, stream);
    else
      e = launch_attend_simt(p.s, cfg->dtype, cache, num_blocks, page_table, max_blocks, B, n_q,
                             p.part, v, seq_lens, di->err, stream);
  }
  if (e == cudaSuccess) {
    if (tc && combine_latent_tc_supported(p.s))
      e = launch_combine_latent_tc(p.s, B, n_q, p.part, v, o_lat, di->err, stream);
    else
      e = launch_combine_latent(p.s, B, n_q, p.part, v, o_lat, stream);
  }
  return from_cuda(e);
}

mla_status mla_quantize_rows_fp8(const mla_config* cfg, const float* rows, const int32_t* seq_idx,
                                 const int32_t* pos, const int32_t* page_table, int32_t B,
                                 int32_t max_blocks, void* cache, float* row_scale,
                                 int32_t num_blocks, int32_t T, cudaStream_t stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (T < 0 || B < 1 || max_blocks < 1 || num_blocks < 1) return MLA_ERR_SHAPE;
  if (T == 0) return MLA_OK;
  if (!rows || !seq_idx || !pos || !page_table || !cache || !row_scale) return MLA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  if (!fp8_supported(cfg, di)) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(cache) || !aligned16(row_scale)) return MLA_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_rows_fp8(shape_of(cfg), rows, seq_idx, pos, page_table, B,
                                            max_blocks, static_cast<uint8_t*>(cache), row_scale,
                                            num_blocks, T, di->err, stream));
}

mla_status mla_append_kv_fp8_workspace_size(const mla_config* cfg, int32_t T, size_t* bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = 0;
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (T < 0) return MLA_ERR_SHAPE;
  const int chunk = T < kFp8AppendChunk ? T : kFp8AppendChunk;
  *bytes = align256(sizeof(float) * static_cast<size_t>(chunk) * shape_of(cfg).R());
  return MLA_OK;
}

mla_status mla_append_kv_fp8(const mla_config* cfg, mla_weights w, const void* x,
                             const int32_t* seq_idx, const int32_t* pos,
                             const int32_t* page_table, int32_t B, int32_t max_blocks,
                             void* cache, float* row_scale, int32_t num_blocks, int32_t T,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!w) return MLA_ERR_INVALID_ARG;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (T < 0 || B < 1 || max_blocks < 1 || num_blocks < 1) return MLA_ERR_SHAPE;
  if (T == 0) return MLA_OK;
  if (!x || !seq_idx || !pos || !page_table || !cache || !row_scale) return MLA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  if (!fp8_supported(cfg, di)) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(cache) || !aligned16(row_scale)) return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_append_kv_fp8_workspace_size(cfg, T, &need);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || ws_bytes < need)
    return MLA_ERR_WORKSPACE;
  const Shape s = shape_of(cfg);
  float* rows = static_cast<float*>(workspace);
  const char* xb = static_cast<const char*>(x);
  const size_t x_row = static_cast<size_t>(s.d_model) * dtype_bytes(cfg->dtype);
  cudaError_t e = cudaSuccess;
  for (int off = 0; off < T && e == cudaSuccess; off += kFp8AppendChunk) {
    const int n = T - off < kFp8AppendChunk ? T - off : kFp8AppendChunk;
    e = launch_append_rows_f32(s, cfg->dtype, &w->w, xb + off * x_row, seq_idx + off, pos + off,
                               n, rows, di->err, stream);
    if (e == cudaSuccess)
      e = launch_quantize_rows_fp8(s, rows, seq_idx + off, pos + off, page_table, B, max_blocks,
                                   static_cast<uint8_t*>(cache), row_scale, num_blocks, n,
                                   di->err, stream);
  }
  return from_cuda(e);
}

mla_status mla_decode_fp8(const mla_config* cfg, mla_weights w, const void* q, const void* cache,
                          const float* row_scale, int32_t num_blocks, const int32_t* page_table,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                          float* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!w || !q || !cache || !row_scale || !page_table || !seq_lens || !out)
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  mla_status st = check_decode_args(cfg, B, n_q);
  if (st != MLA_OK) return st;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  if (!fp8_supported(cfg, di)) return MLA_ERR_UNSUPPORTED;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(row_scale)) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * cfg->block_size > (1LL << 31) - 1) return MLA_ERR_SHAPE;
  Plan p;
  make_plan(cfg, B, n_q, di, MLA_IMPL_TENSOR_CORE, &p);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MLA_ERR_WORKSPACE;
  if (ws_bytes < p.lay.total) return MLA_ERR_WORKSPACE;
  const WsView v = ws_view(workspace, p.lay);
  // fp16 queries, pre-multiplied by scale * log2(e) as for the bf16 kernel
  cudaError_t e = launch_absorb_q_tc(p.s, &w->w, q, seq_lens, max_blocks, B, n_q, p.part, v,
                                     p.s.scale * 1.4426950408889634f, true, di->err, stream);
  if (e == cudaSuccess)
    e = launch_attend_tc_fp8(p.s, cache, row_scale, num_blocks, page_table, max_blocks, B, n_q,
                             p.part, v, seq_lens, di->err, stream);
  if (e == cudaSuccess)
    e = aligned16(out)
            ? launch_combine_tc(p.s, &w->w, B, n_q, p.part, v, out, nullptr, di->err, stream)
            : launch_combine(p.s, cfg->dtype, &w->w, seq_lens, B, n_q, p.part, v, out, stream);
  return from_cuda(e);
}

mla_status mla_fold_full(const mla_config* cfg, const void* W_q, const void* W_uk,
                         const void* W_uv, const void* W_o, cudaStream_t stream,
                         mla_full_weights* out) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  mla_status st = check_config(cfg);
  if (st != MLA_OK) return st;
  if (!W_q || !W_uk || !W_uv || !W_o) return MLA_ERR_INVALID_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  const int dev = current_device();
  const Shape s = shape_of(cfg);
  const size_t n_qf = sizeof(float) * static_cast<size_t>(s.d_model) * s.n_h * s.R();
  const size_t n_vo = sizeof(float) * static_cast<size_t>(s.n_h) * s.d_c * s.d_model;
  const int half = s.d_r / 2;
  mla_full_weights_s* h = new (std::nothrow) mla_full_weights_s();
  if (!h) return MLA_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->w.shape = s;
  h->w.dtype = cfg->dtype;
  h->w.device = dev;
  auto release = [h]() {
    cudaFree(h->w.w_qf);
    cudaFree(h->w.w_vo);
    cudaFree(h->w.rope_turns);
    delete h;
  };
  if (cudaMalloc(&h->w.w_qf, n_qf) != cudaSuccess || cudaMalloc(&h->w.w_vo, n_vo) != cudaSuccess ||
      cudaMalloc(&h->w.rope_turns, sizeof(uint64_t) * half) != cudaSuccess) {
    cudaGetLastError();
    release();
    return MLA_ERR_CUDA;
  }
  uint64_t turns[512];
  rope_turn_table(cfg->rope_base, s.d_r, turns);
  cudaError_t e = cudaMemcpyAsync(h->w.rope_turns, turns, sizeof(uint64_t) * half,
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess)
    e = launch_fold_full(s, cfg->dtype, W_q, W_uk, W_uv, W_o, &h->w, di->sms, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaStreamSynchronize(stream);
    release();
    return MLA_ERR_CUDA;
  }
  *out = h;
  return MLA_OK;
}

mla_status mla_full_weights_free(mla_full_weights w) {
  if (!w) return MLA_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(w->w.device);
  cudaDeviceSynchronize();
  cudaFree(w->w.w_qf);
  cudaFree(w->w.w_vo);
  cudaFree(w->w.rope_turns);
  if (prev >= 0) cudaSetDevice(prev);
  delete w;
  return MLA_OK;
}

mla_status mla_decode_full_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                          size_t* bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = 0;
  size_t base = 0;
  mla_status st = mla_decode_workspace_size(cfg, B, n_q, 0, &base);
  if (st != MLA_OK) return st;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  *bytes = base + full_extra(shape_of(cfg), B, n_q, di->sms).total;
  return MLA_OK;
}

mla_status mla_decode_full(const mla_config* cfg, mla_full_weights fw, const void* x_q,
                           const void* cache, int32_t num_blocks, const int32_t* page_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                           float* y, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!fw || !x_q || !cache || !page_table || !seq_lens || !y) return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, cache, workspace, ws_bytes, &p, &di, true);
  if (st != MLA_OK) return st;
  if (!same_shape(cfg, &fw->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != fw->w.device) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * cfg->block_size > (1LL << 31) - 1) return MLA_ERR_SHAPE;
  const FullExtra fx = full_extra(p.s, B, n_q, di->sms);
  if (ws_bytes < p.lay.total + fx.total) return MLA_ERR_WORKSPACE;
  const WsView v = ws_view(workspace, p.lay);
  float* proj = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.lay.total);
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.lay.total + fx.proj);
  const int M = B * n_q;
  // 1. x_q [W_abs[h] | W_qr[h]] for every head, then RoPE, scale, rounding and the plan
  cudaError_t e = launch_xw(cfg->dtype, x_q, M, p.s.d_model, MLA_F32, fw->w.w_qf,
                            p.s.n_h * p.s.R(), proj, part, fx.q, di->err, false, stream);
  const float out_scale =
      p.impl == MLA_IMPL_TENSOR_CORE ? p.s.scale * 1.4426950408889634f : 1.f;
  if (e == cudaSuccess)
    e = launch_q_finish(p.s, cfg->dtype, fw->w.rope_turns, proj, seq_lens, max_blocks, B, n_q,
                        p.part, v, out_scale, p.impl == MLA_IMPL_CUDA_CORE, di->err, stream);
  // 2. split-KV latent attention, the same kernels as mla_decode
  if (e == cudaSuccess) {
    if (p.impl == MLA_IMPL_TENSOR_CORE)
      e = launch_attend_tc(p.s, cache, num_blocks, page_table, max_blocks, B, n_q, p.part, v,
                           seq_lens, di->err, stream);
    else
      e = launch_attend_simt(p.s, cfg->dtype, cache, num_blocks, page_table, max_blocks, B, n_q,
                             p.part, v, seq_lens, di->err, stream);
  }
  // 3. merge the splits into o_lat (over the projection, which is spent)
  if (e == cudaSuccess) e = launch_combine_latent(p.s, B, n_q, p.part, v, proj, stream);
  // 4. y = sum_h o_lat[h] W_vo[h]
  if (e == cudaSuccess)
    e = launch_xw(MLA_F32, proj, M, p.s.n_h * p.s.d_c, MLA_F32, fw->w.w_vo, p.s.d_model, y,
                  part, fx.o, di->err, false, stream);
  return from_cuda(e);
}

namespace {

// Workspace of mla_decode_layer past the decode's own: the bf16 hi/lo copy
// of out that the tensor-core projection reads (decode-sized batches only),
// then the projection's split partials, sized for either projection kernel.
struct LayerExtra {
  size_t hilo_bytes, part_bytes;
  XwPlan po, pp;  // K splits of the CUDA-core and the tensor-core projection
};
LayerExtra layer_extra(const mla_config* cfg, int M, const DeviceInfo* di) {
  const int K = cfg->n_h * cfg->d_v, N = cfg->d_model;
  LayerExtra x;
  x.po = xw_plan(M, K, N, di->sms);
  size_t floats = xw_part_floats(M, N, x.po);
  x.hilo_bytes = 0;
  x.pp = x.po;
  if (M <= PROJ_TC_MAX_TOKENS) {
    x.hilo_bytes = align256(sizeof(uint16_t) * 2 * static_cast<size_t>(M) * K);
    x.pp = proj_tc_plan(M, K, N, di->sms);
    if (x.pp.S > 1) floats = std::max(floats, static_cast<size_t>(x.pp.S) * M * N);
  }
  x.part_bytes = align256(sizeof(float) * floats);
  return x;
}

}  // namespace

mla_status mla_decode_layer_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                           size_t* bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  *bytes = 0;
  size_t base = 0;
  mla_status st = mla_decode_workspace_size(cfg, B, n_q, 0, &base);
  if (st != MLA_OK) return st;
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  const LayerExtra x = layer_extra(cfg, B * n_q, di);
  *bytes = base + x.hilo_bytes + x.part_bytes;
  return MLA_OK;
}

mla_status mla_decode_layer(const mla_config* cfg, mla_weights w, const void* W_o, const void* x,
                            const int32_t* seq_idx, const int32_t* pos, const void* q,
                            void* cache, int32_t num_blocks, const int32_t* page_table,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                            float* out, float* y, void* workspace, size_t ws_bytes,
                            cudaStream_t stream) {
  if (!w || !W_o || !x || !seq_idx || !pos || !q || !cache || !page_table || !seq_lens || !out ||
      !y)
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks < 1) return MLA_ERR_SHAPE;
  Plan p;
  const DeviceInfo* di = nullptr;
  mla_status st = prepare_decode(cfg, B, n_q, cache, workspace, ws_bytes, &p, &di, true);
  if (st != MLA_OK) return st;
  if (!same_shape(cfg, &w->cfg)) return MLA_ERR_SHAPE;
  if (current_device() != w->w.device) return MLA_ERR_INVALID_ARG;
  const int M = B * n_q, K = p.s.n_h * p.s.d_v, N = p.s.d_model;
  const LayerExtra xl = layer_extra(cfg, M, di);
  if (ws_bytes < p.lay.total + xl.hilo_bytes + xl.part_bytes) return MLA_ERR_WORKSPACE;
  char* extra = static_cast<char*>(workspace) + p.lay.total;
  uint16_t* hilo = reinterpret_cast<uint16_t*>(extra);
  float* part = reinterpret_cast<float*>(extra + xl.hilo_bytes);
  // The new tokens go into the cache first, then the decode reads them.
  st = mla_append_kv(cfg, w, x, seq_idx, pos, page_table, B, max_blocks, cache, num_blocks, M,
                     stream);
  if (st != MLA_OK) return st;
  // The tensor-core projection takes out from the tensor-core combine as a
  // bf16 hi/lo pair; every other case projects out (fp32) on the CUDA cores.
  const bool tc = p.impl == MLA_IMPL_TENSOR_CORE && combine_tc_supported(p.s, cfg->dtype) &&
                  aligned16(out) && xl.hilo_bytes > 0 && proj_tc_applies(M, K, N, W_o);
  if (!tc) {
    st = mla_decode(cfg, w, q, cache, num_blocks, page_table, max_blocks, seq_lens, B, n_q, out,
                    workspace, ws_bytes, stream);
    if (st != MLA_OK) return st;
    // y = concat_h(o_h) W_o, launched early: its W_o stream overlaps the combine
    return from_cuda(launch_xw(MLA_F32, out, M, K, cfg->dtype, W_o, N, y, part, xl.po, di->err,
                               true, stream));
  }
  mla_config c2 = *cfg;
  c2.impl = p.impl;
  st = mla_decode_absorb_q(&c2, w, q, seq_lens, max_blocks, B, n_q, workspace, ws_bytes, stream);
  if (st != MLA_OK) return st;
  st = mla_decode_attend(&c2, cache, num_blocks, page_table, max_blocks, seq_lens, B, n_q,
                         workspace, ws_bytes, stream);
  if (st != MLA_OK) return st;
  const WsView v = ws_view(workspace, p.lay);
  cudaError_t e = launch_combine_tc(p.s, &w->w, B, n_q, p.part, v, out, hilo, di->err, stream);
  // y = concat_h(o_h) W_o on the tensor cores, launched early: its W_o
  // stream overlaps the combine
  if (e == cudaSuccess) e = launch_proj_tc(hilo, M, K, W_o, N, y, part, xl.pp, di->err, stream);
  return from_cuda(e);
}

mla_status mla_get_last_device_error(cudaStream_t stream, uint32_t* code) {
  if (!code) return MLA_ERR_INVALID_ARG;
  *code = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  const DeviceInfo* di = device_info();
  if (!di) return MLA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mla_device_error, sizeof(v)) != cudaSuccess) return MLA_ERR_CUDA;
  if (v) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_mla_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  *code = v;
  if (v & MLA_DEVERR_TIMEOUT) return MLA_ERR_TIMEOUT;
  return v ? MLA_ERR_DEVICE_CHECK : MLA_OK;
}

}  // extern "C"
