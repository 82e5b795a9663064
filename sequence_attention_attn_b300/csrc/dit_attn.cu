// dit_attn.cu -- the C ABI of libditattn.so (declared in include/dit_attn.h):
// argument validation, TMA descriptor encoding and kernel launches.
//
// Every check that can be made without the GPU is made first, so invalid
// calls return an error code before any CUDA call.  Tensor maps are encoded
// on the host through the driver entry point fetched by the runtime (no link
// against libcuda).  Nothing is allocated on any call path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "dit_attn.h"
#include "attn_fwd.cuh"
#include "cfg_static.cuh"
#include "merge_cfg.cuh"
#include "ptx.cuh"

namespace {

constexpr int kAbiVersion = 2;
constexpr int kMaxDevices = 64;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

constexpr int kMaxTorusChunks = 64;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
  // Events of the Torus pipeline (created on first use, reused by every call).
  cudaEvent_t torus_events[kMaxTorusChunks + 1] = {};
  bool torus_events_ready = false;
  bool attr_set[3][2][2][2] = {};  // per head-dim instantiation x partials x programmatic launch x grid walk
};

std::mutex g_mu;
// Device address of the rel-MAE scratch array (cfg_static.cuh), looked up on
// the first cfg_combine_relmae_static call on each device, with it current.
double *g_relmae_scratch_ptr[kMaxDevices] = {};
// Serialises dit_attn_fwd_torus calls: they share one event pool per device.
std::mutex g_torus_mu;
// Serialises status reads: they share the device word the exchange writes to.
std::mutex g_status_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Makes the stream's device current for this library's runtime and checks
// that it is an sm_103 part.
dit_status select_device(dit_stream_t stream, int *dev_out, DeviceState **st_out) {
  int dev = 0;
  cudaError_t e;
  if (stream != nullptr) {
    e = cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &dev);
    if (e != cudaSuccess) return DIT_ERR_CUDA;
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return DIT_ERR_CUDA;
  } else {
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return DIT_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DIT_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &st = g_dev[dev];
  if (!st.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DIT_ERR_CUDA;
    st.probed = true;
    st.supported = (major == 10 && minor == 3);
    st.sm_count = sms;
  }
  if (!st.supported) return DIT_ERR_UNSUPPORTED_DEVICE;
  *dev_out = dev;
  *st_out = &st;
  return DIT_OK;
}

dit_status get_encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode != nullptr) return DIT_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return DIT_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return DIT_OK;
}

// 3-D bf16 view [BH][rows][D] of one of q, k, v (head stride S rows); a box
// of `box_cols` x 128 rows.  Rows >= `rows` of a head are never read: TMA
// fills them with zeros.
dit_status encode_qkv_map(CUtensorMap *map, const void *ptr, long long BH, int S, int rows, int D, int box_cols,
                          CUtensorMapSwizzle swz) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(ditk::kBlockM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DIT_OK : DIT_ERR_CUDA;
}

// bf16 [BH][S][D] output as a TMA store target: a box of all D columns by 32
// rows, no swizzle (rows of D * 2 bytes, packed).
dit_status encode_out_map(CUtensorMap *map, void *ptr, long long BH, int S, int D) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DIT_OK : DIT_ERR_CUDA;
}

// Launches a kernel with programmatic stream serialization: it may start
// while the previous kernel in the stream finishes, and waits for it (in the
// kernel, griddep_wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int head_dim_index(int D) { return D == 64 ? 0 : (D == 72 ? 1 : (D == 128 ? 2 : -1)); }

dit_status check_attn_args(const void *q, const void *k, const void *v, int B, int H, int S, int D, int n) {
  if (q == nullptr || k == nullptr || v == nullptr) return DIT_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || n < 1 || n > S) return DIT_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 2147483647LL) return DIT_ERR_INVALID_ARG;
  if (head_dim_index(D) < 0) return DIT_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return DIT_ERR_MISALIGNED;
  return DIT_OK;
}

// Grids of up to this many waves (one CTA per SM) take the programmatic
// launch: the next kernel's CTAs start on the SMs this one leaves idle.
constexpr int kPdlMaxWaves = 8;

template <int D, bool kPartials>
dit_status launch_attn(DeviceState &st, int didx, const void *q, const void *k, const void *v,
                       const ditk::AttnParams &prm, long long BH, int S, int grid, cudaStream_t stream,
                       bool grid_walk) {
  using L = ditk::AttnLayout<D>;
  const bool pdl = grid <= kPdlMaxWaves * st.sm_count;
  auto kernel = pdl ? ditk::attn_fwd_kernel<D, kPartials, true> : ditk::attn_fwd_kernel<D, kPartials, false>;
  if constexpr (!kPartials && D == 128) {
    if (grid_walk)
      kernel = pdl ? ditk::attn_fwd_kernel<D, false, true, true> : ditk::attn_fwd_kernel<D, false, false, true>;
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    bool &done = st.attr_set[didx][kPartials ? 1 : 0][pdl ? 1 : 0][grid_walk ? 1 : 0];
    if (!done) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemLaunch) !=
          cudaSuccess)
        return DIT_ERR_CUDA;
      done = true;
    }
  }
  CUtensorMap mq, mq_t, mk, mk_t, mv, mv_t;
  dit_status s;
  // A key range [j0, j1) maps only the key rows below j1, so the masked tail
  // of its last tile is zero-filled by TMA instead of read.
  const int kv_rows = prm.key_j1 > 0 ? prm.key_j1 : S;
  if ((s = encode_qkv_map(&mq, q, BH, S, S, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != DIT_OK) return s;
  if ((s = encode_qkv_map(&mk, k, BH, S, kv_rows, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != DIT_OK) return s;
  if ((s = encode_qkv_map(&mv, v, BH, S, kv_rows, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != DIT_OK) return s;
  // Columns 64.. of Q and K: a 16-column 32-byte-swizzled box for D = 72 (the
  // last K step of QK^T), the main map's 64-column box otherwise.  V always
  // takes the main map's box at column 64 (D = 72: columns 72..127 of that box
  // are zero-filled, and PV runs with N = 80).
  if (D == 72) {
    if ((s = encode_qkv_map(&mq_t, q, BH, S, S, D, 16, CU_TENSOR_MAP_SWIZZLE_32B)) != DIT_OK) return s;
    if ((s = encode_qkv_map(&mk_t, k, BH, S, kv_rows, D, 16, CU_TENSOR_MAP_SWIZZLE_32B)) != DIT_OK) return s;
  } else {
    mq_t = mq;
    mk_t = mk;
  }
  mv_t = mv;
  // The output as a TMA store target (merged mode at D = 72; the other
  // instantiations never read this parameter).
  CUtensorMap mo = mq;
  if (!kPartials && D == 72 && (s = encode_out_map(&mo, prm.out, BH, S, D)) != DIT_OK) return s;
  if (pdl) {
    if (launch_pdl(kernel, dim3(grid), dim3(ditk::kAttnThreads), L::kSmemLaunch, stream, mq, mq_t, mk, mk_t, mv,
                   mv_t, mo, prm) != cudaSuccess)
      return DIT_ERR_LAUNCH;
  } else {
    kernel<<<grid, ditk::kAttnThreads, L::kSmemLaunch, stream>>>(mq, mq_t, mk, mk_t, mv, mv_t, mo, prm);
  }
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

// key_j1 > 0 (partials mode only): one key range [key_j0, key_j1), written
// to the first partial slot.
template <bool kPartials>
dit_status attn_dispatch(const void *q, const void *k, const void *v, void *out, float *lse, float *partials,
                         float *part_lse, int B, int H, int S, int D, int n, dit_stream_t stream, int key_j0 = 0,
                         int key_j1 = 0) {
  const long long BH = static_cast<long long>(B) * H;
  const int tiles_q = (S + ditk::kBlockM - 1) / ditk::kBlockM;
  const int num_pairs = (tiles_q + 1) / 2;
  long long grid = BH * num_pairs * (kPartials ? n : 1);
  if (grid > 2147483647LL) return DIT_ERR_INVALID_ARG;
  long long pair_units = grid;
  // Key tiles over all chunks (each chunk starts a new tile).
  long long tiles_total = 0;
  for (int c = 0; c < n; ++c) {
    const long long j0 = (static_cast<long long>(c) * S) / n, j1 = (static_cast<long long>(c + 1) * S) / n;
    tiles_total += (j1 - j0 + ditk::kBlockN - 1) / ditk::kBlockN;
  }
  // The grid walk (tiles on the global 128-key grid, a chunk end inside a tile
  // splitting only that tile's row sum) for the merged launch at D = 128 when
  // every chunk is at least one tile long and the chunk-by-chunk walk would
  // cut tiles: there the tensor pipe paces the kernel and the cut tiles' MMA
  // work is what the grid walk saves (Flux at 8 chunks: +6 %).  Elsewhere the
  // chunk-by-chunk walk is as fast or faster.
  const long long tiles_grid = (S + ditk::kBlockN - 1) / ditk::kBlockN;
  const bool grid_walk = !kPartials && D == 128 && n > 1 && S / n >= ditk::kBlockN && tiles_total > tiles_grid;
  if (grid_walk) tiles_total = tiles_grid;
  if (tiles_total > 2147483647LL) return DIT_ERR_INVALID_ARG;

  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  if ((s = get_encoder()) != DIT_OK) return s;
  if (!kPartials) {
    // A last wave of at most half the SMs: its pairs run as two single-tile
    // CTAs each, on twice as many SMs.
    const long long rem = grid % st->sm_count;
    if (grid > st->sm_count && rem > 0 && 2 * rem <= st->sm_count) {
      pair_units = grid - rem;
      grid += rem;
    }
  }

  ditk::AttnParams prm{};
  prm.out = static_cast<__nv_bfloat16 *>(out);
  prm.lse = lse;
  prm.partials = partials;
  prm.part_lse = part_lse;
  prm.rows_total = BH * S;
  prm.S = S;
  prm.n_chunks = n;
  prm.num_pairs = num_pairs;
  prm.tiles_total = static_cast<int>(tiles_total);
  prm.key_j0 = key_j0;
  prm.key_j1 = key_j1;
  prm.pair_units = static_cast<int>(pair_units);
  prm.chunk_q = S / n;
  prm.chunk_r = S % n;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  switch (D) {
    case 64:
      return launch_attn<64, kPartials>(*st, 0, q, k, v, prm, BH, S, static_cast<int>(grid), cs, grid_walk);
    case 72:
      return launch_attn<72, kPartials>(*st, 1, q, k, v, prm, BH, S, static_cast<int>(grid), cs, grid_walk);
    default:
      return launch_attn<128, kPartials>(*st, 2, q, k, v, prm, BH, S, static_cast<int>(grid), cs, grid_walk);
  }
}

// Workspace of dit_attn_fwd_split: fp32 partials [n][rows][D], then their
// LSEs [n][rows] from the next 256-byte boundary.
struct SplitWorkspace {
  size_t lse_off, total;
};
SplitWorkspace split_workspace(long long rows, int D, int n) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SplitWorkspace w;
  w.lse_off = up(static_cast<size_t>(n) * rows * D * 4);
  w.total = w.lse_off + up(static_cast<size_t>(n) * rows * 4);
  return w;
}

int stream_grid(const DeviceState &st, long long work_items) {
  const long long per_wave = static_cast<long long>(st.sm_count) * 8;
  const long long need = (work_items + ditk::kStreamThreads - 1) / ditk::kStreamThreads;
  long long g = need < per_wave ? need : per_wave;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

int dit_abi_version(void) { return kAbiVersion; }

const char *dit_status_string(dit_status status) {
  switch (status) {
    case DIT_OK:
      return "ok";
    case DIT_ERR_INVALID_ARG:
      return "invalid argument (null pointer, bad size, count or aliasing)";
    case DIT_ERR_UNSUPPORTED_SHAPE:
      return "unsupported shape (head dimension must be 64, 72 or 128)";
    case DIT_ERR_MISALIGNED:
      return "pointer not 16-byte aligned";
    case DIT_ERR_UNSUPPORTED_DEVICE:
      return "unsupported device (needs compute capability 10.3, B300)";
    case DIT_ERR_LAUNCH:
      return "kernel launch failed";
    case DIT_ERR_DEVICE_TIMEOUT:
      return "a bounded device-side wait ran out; results are invalid";
    case DIT_ERR_CUDA:
      return "CUDA runtime or driver error";
  }
  return "unknown status";
}

dit_status dit_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                        int S, int D, int n_kv_chunks, dit_stream_t stream) {
  dit_status s = check_attn_args(q, k, v, B, H, S, D, n_kv_chunks);
  if (s != DIT_OK) return s;
  if (out == nullptr) return DIT_ERR_INVALID_ARG;
  if (!aligned16(out) || (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
    return DIT_ERR_MISALIGNED;
  const size_t bytes = static_cast<size_t>(B) * H * S * D * 2;
  if (ranges_overlap(out, bytes, q, bytes) || ranges_overlap(out, bytes, k, bytes) ||
      ranges_overlap(out, bytes, v, bytes))
    return DIT_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const size_t lb = static_cast<size_t>(B) * H * S * 4;
    if (ranges_overlap(lse, lb, q, bytes) || ranges_overlap(lse, lb, k, bytes) ||
        ranges_overlap(lse, lb, v, bytes) || ranges_overlap(lse, lb, out, bytes))
      return DIT_ERR_INVALID_ARG;
  }
  return attn_dispatch<false>(q, k, v, out, lse, nullptr, nullptr, B, H, S, D, n_kv_chunks, stream);
}

dit_status dit_attn_fwd_partials(const void *q, const void *k, const void *v, float *partials, float *lses,
                                 int B, int H, int S, int D, int n_kv_chunks, dit_stream_t stream) {
  dit_status s = check_attn_args(q, k, v, B, H, S, D, n_kv_chunks);
  if (s != DIT_OK) return s;
  if (partials == nullptr || lses == nullptr) return DIT_ERR_INVALID_ARG;
  if (!aligned16(partials) || !aligned16(lses)) return DIT_ERR_MISALIGNED;
  const size_t in_bytes = static_cast<size_t>(B) * H * S * D * 2;
  const size_t p_bytes = static_cast<size_t>(n_kv_chunks) * B * H * S * D * 4;
  const size_t l_bytes = static_cast<size_t>(n_kv_chunks) * B * H * S * 4;
  if (ranges_overlap(partials, p_bytes, q, in_bytes) || ranges_overlap(partials, p_bytes, k, in_bytes) ||
      ranges_overlap(partials, p_bytes, v, in_bytes) || ranges_overlap(lses, l_bytes, q, in_bytes) ||
      ranges_overlap(lses, l_bytes, k, in_bytes) || ranges_overlap(lses, l_bytes, v, in_bytes) ||
      ranges_overlap(lses, l_bytes, partials, p_bytes))
    return DIT_ERR_INVALID_ARG;
  return attn_dispatch<true>(q, k, v, nullptr, nullptr, partials, lses, B, H, S, D, n_kv_chunks, stream);
}

// The merge kernel's size limits: rows * D < 2^40, n * rows * D <= 2^46.
bool split_sizes_ok(long long rows, int D, int n) {
  return rows <= (1LL << 40) / D && static_cast<long long>(n) * rows * D <= (1LL << 46);
}

size_t dit_attn_split_workspace_bytes(int B, int H, int S, int D, int n_split) {
  if (B < 1 || H < 1 || S < 1 || n_split < 1 || n_split > S || head_dim_index(D) < 0) return 0;
  if (static_cast<long long>(B) * H > 2147483647LL) return 0;
  const long long rows = static_cast<long long>(B) * H * S;
  if (!split_sizes_ok(rows, D, n_split)) return 0;
  return split_workspace(rows, D, n_split).total;
}

dit_status dit_attn_fwd_split(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                              int S, int D, int n_split, void *workspace, size_t workspace_bytes,
                              dit_stream_t stream) {
  dit_status s = check_attn_args(q, k, v, B, H, S, D, n_split);
  if (s != DIT_OK) return s;
  if (out == nullptr || workspace == nullptr) return DIT_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(workspace) || (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
    return DIT_ERR_MISALIGNED;
  const long long rows = static_cast<long long>(B) * H * S;
  if (!split_sizes_ok(rows, D, n_split)) return DIT_ERR_INVALID_ARG;
  const SplitWorkspace w = split_workspace(rows, D, n_split);
  if (workspace_bytes < w.total) return DIT_ERR_INVALID_ARG;
  const size_t bytes = static_cast<size_t>(rows) * D * 2, lb = static_cast<size_t>(rows) * 4;
  const void *inputs[] = {q, k, v};
  for (const void *b : inputs) {
    if (ranges_overlap(out, bytes, b, bytes) || ranges_overlap(workspace, w.total, b, bytes) ||
        (lse != nullptr && ranges_overlap(lse, lb, b, bytes)))
      return DIT_ERR_INVALID_ARG;
  }
  if (ranges_overlap(workspace, w.total, out, bytes) ||
      (lse != nullptr && (ranges_overlap(lse, lb, out, bytes) || ranges_overlap(lse, lb, workspace, w.total))))
    return DIT_ERR_INVALID_ARG;
  float *partials = static_cast<float *>(workspace);
  float *lses = reinterpret_cast<float *>(static_cast<char *>(workspace) + w.lse_off);
  // One CTA per (query-tile pair, chunk): each chunk's normalised partial
  // and LSE to the workspace ...
  if ((s = attn_dispatch<true>(q, k, v, nullptr, nullptr, partials, lses, B, H, S, D, n_split, stream)) != DIT_OK)
    return s;
  // ... then their log-sum-exp merge over all rows, rounded to bf16 (a
  // programmatic launch: it starts as the attention CTAs finish and waits
  // for all of them before reading the workspace).
  int dev = 0;
  DeviceState *st = nullptr;
  if ((s = select_device(stream, &dev, &st)) != DIT_OK) return s;
  const int d4 = D / 4;
  if (launch_pdl(ditk::lse_merge_bf16_kernel, dim3(stream_grid(*st, rows * d4)), dim3(ditk::kStreamThreads), 0,
                 reinterpret_cast<cudaStream_t>(stream), static_cast<const float *>(partials),
                 static_cast<const float *>(lses), n_split, static_cast<__nv_bfloat16 *>(out), lse, rows,
                 d4) != cudaSuccess)
    return DIT_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status dit_attn_fwd_range(const void *q, const void *k, const void *v, float *out, float *lse, int B, int H,
                              int S, int D, int j0, int j1, dit_stream_t stream) {
  dit_status s = check_attn_args(q, k, v, B, H, S, D, 1);
  if (s != DIT_OK) return s;
  if (out == nullptr || lse == nullptr) return DIT_ERR_INVALID_ARG;
  if (j0 < 0 || j1 > S || j0 >= j1) return DIT_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(lse)) return DIT_ERR_MISALIGNED;
  const size_t in_bytes = static_cast<size_t>(B) * H * S * D * 2;
  const size_t o_bytes = static_cast<size_t>(B) * H * S * D * 4;
  const size_t l_bytes = static_cast<size_t>(B) * H * S * 4;
  if (ranges_overlap(out, o_bytes, q, in_bytes) || ranges_overlap(out, o_bytes, k, in_bytes) ||
      ranges_overlap(out, o_bytes, v, in_bytes) || ranges_overlap(lse, l_bytes, q, in_bytes) ||
      ranges_overlap(lse, l_bytes, k, in_bytes) || ranges_overlap(lse, l_bytes, v, in_bytes) ||
      ranges_overlap(lse, l_bytes, out, o_bytes))
    return DIT_ERR_INVALID_ARG;
  return attn_dispatch<true>(q, k, v, nullptr, nullptr, out, lse, B, H, S, D, 1, stream, j0, j1);
}

dit_status dit_attn_fwd_torus(const void *q, const void *k_src, const void *v_src, void *k, void *v,
                              float *partials, float *lses, float *out, float *lse_out, int B, int H, int S, int D,
                              int n_kv_chunks, dit_stream_t stream, dit_stream_t copy_stream) {
  const int n = n_kv_chunks;
  dit_status s = check_attn_args(q, k, v, B, H, S, D, n);
  if (s != DIT_OK) return s;
  if (n > kMaxTorusChunks) return DIT_ERR_INVALID_ARG;
  if (k_src == nullptr || v_src == nullptr || partials == nullptr || lses == nullptr || out == nullptr)
    return DIT_ERR_INVALID_ARG;
  if (!aligned16(partials) || !aligned16(lses) || !aligned16(out) || (lse_out != nullptr && !aligned16(lse_out)))
    return DIT_ERR_MISALIGNED;
  const long long BH = static_cast<long long>(B) * H;
  const long long rows = BH * S;
  const size_t kv_bytes = static_cast<size_t>(rows) * D * 2;
  const size_t p_bytes = static_cast<size_t>(n) * rows * D * 4, l_bytes = static_cast<size_t>(n) * rows * 4;
  const size_t o_bytes = static_cast<size_t>(rows) * D * 4;
  const void *dev_bufs[] = {q, k, v};
  for (const void *b : dev_bufs) {
    if (ranges_overlap(partials, p_bytes, b, kv_bytes) || ranges_overlap(lses, l_bytes, b, kv_bytes) ||
        ranges_overlap(out, o_bytes, b, kv_bytes))
      return DIT_ERR_INVALID_ARG;
  }
  if (ranges_overlap(k, kv_bytes, v, kv_bytes) || ranges_overlap(k, kv_bytes, q, kv_bytes) ||
      ranges_overlap(v, kv_bytes, q, kv_bytes) || ranges_overlap(k_src, kv_bytes, k, kv_bytes) ||
      ranges_overlap(v_src, kv_bytes, v, kv_bytes) || ranges_overlap(k_src, kv_bytes, v, kv_bytes) ||
      ranges_overlap(v_src, kv_bytes, k, kv_bytes) || ranges_overlap(lses, l_bytes, partials, p_bytes))
    return DIT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState *st = nullptr;
  if ((s = select_device(stream, &dev, &st)) != DIT_OK) return s;
  std::lock_guard<std::mutex> torus_lock(g_torus_mu);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st->torus_events_ready) {
      for (int i = 0; i <= kMaxTorusChunks; ++i)
        if (cudaEventCreateWithFlags(&st->torus_events[i], cudaEventDisableTiming) != cudaSuccess)
          return DIT_ERR_CUDA;
      st->torus_events_ready = true;
    }
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t xs = copy_stream != nullptr ? reinterpret_cast<cudaStream_t>(copy_stream) : cs;
  cudaEvent_t *ev = st->torus_events;
  // The copies may only overwrite k and v once the work queued before this
  // call on the compute stream (which may still read them) is done.
  if (xs != cs) {
    if (cudaEventRecord(ev[kMaxTorusChunks], cs) != cudaSuccess) return DIT_ERR_CUDA;
    if (cudaStreamWaitEvent(xs, ev[kMaxTorusChunks], 0) != cudaSuccess) return DIT_ERR_CUDA;
  }
  const size_t pitch = static_cast<size_t>(S) * D * 2;
  auto bound = [&](int c) { return static_cast<int>((static_cast<long long>(c) * S) / n); };
  // Chunk c's key rows of every (batch, head): one strided copy per tensor.
  for (int c = 0; c < n; ++c) {
    const size_t off = static_cast<size_t>(bound(c)) * D * 2, width = static_cast<size_t>(bound(c + 1) - bound(c)) * D * 2;
    if (cudaMemcpy2DAsync(static_cast<char *>(k) + off, pitch, static_cast<const char *>(k_src) + off, pitch, width,
                          static_cast<size_t>(BH), cudaMemcpyDefault, xs) != cudaSuccess ||
        cudaMemcpy2DAsync(static_cast<char *>(v) + off, pitch, static_cast<const char *>(v_src) + off, pitch, width,
                          static_cast<size_t>(BH), cudaMemcpyDefault, xs) != cudaSuccess)
      return DIT_ERR_CUDA;
    if (cudaEventRecord(ev[c], xs) != cudaSuccess) return DIT_ERR_CUDA;
  }
  // Chunk c is computed as soon as its own rows have arrived: the key-range
  // kernel reads no row at or past the chunk end (TMA zero-fills the tail of
  // its last tile), so later chunks may still be in flight.
  for (int c = 0; c < n; ++c) {
    const long long j0 = bound(c), j1 = bound(c + 1);
    if (cudaStreamWaitEvent(cs, ev[c], 0) != cudaSuccess) return DIT_ERR_CUDA;
    s = attn_dispatch<true>(q, k, v, nullptr, nullptr, partials + static_cast<size_t>(c) * rows * D,
                            lses + static_cast<size_t>(c) * rows, B, H, S, D, 1, stream, static_cast<int>(j0),
                            static_cast<int>(j1));
    if (s != DIT_OK) return s;
  }
  return dit_attn_merge(partials, lses, n, out, lse_out, rows, D, stream);
}

dit_status dit_attn_merge(const float *partials, const float *lses, int n, float *out, float *lse_out,
                          long long rows, int D, dit_stream_t stream) {
  if (partials == nullptr || lses == nullptr || out == nullptr) return DIT_ERR_INVALID_ARG;
  if (n < 1 || rows < 1 || D < 1) return DIT_ERR_INVALID_ARG;
  if (rows > (1LL << 40) / D || static_cast<long long>(n) * rows * D > (1LL << 46))
    return DIT_ERR_INVALID_ARG;
  if (!aligned16(partials) || !aligned16(lses) || !aligned16(out) ||
      (lse_out != nullptr && !aligned16(lse_out)))
    return DIT_ERR_MISALIGNED;
  const size_t p_bytes = static_cast<size_t>(n) * rows * D * 4, l_bytes = static_cast<size_t>(n) * rows * 4;
  const size_t o_bytes = static_cast<size_t>(rows) * D * 4, lo_bytes = static_cast<size_t>(rows) * 4;
  if (ranges_overlap(out, o_bytes, partials, p_bytes) || ranges_overlap(out, o_bytes, lses, l_bytes))
    return DIT_ERR_INVALID_ARG;
  if (lse_out != nullptr &&
      (ranges_overlap(lse_out, lo_bytes, partials, p_bytes) || ranges_overlap(lse_out, lo_bytes, lses, l_bytes) ||
       ranges_overlap(lse_out, lo_bytes, out, o_bytes)))
    return DIT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (D % 4 == 0) {
    const int d4 = D / 4;
    if (launch_pdl(ditk::lse_merge_vec4_kernel, dim3(stream_grid(*st, rows * d4)), dim3(ditk::kStreamThreads), 0, cs,
                   partials, lses, n, out, lse_out, rows, d4) != cudaSuccess)
      return DIT_ERR_LAUNCH;
  } else {
    if (launch_pdl(ditk::lse_merge_scalar_kernel, dim3(stream_grid(*st, rows * D)), dim3(ditk::kStreamThreads), 0, cs,
                   partials, lses, n, out, lse_out, rows, D) != cudaSuccess)
      return DIT_ERR_LAUNCH;
  }
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status cfg_combine(const float *eps_c, const float *eps_u, float w, float *out, long long numel,
                       dit_stream_t stream) {
  if (eps_c == nullptr || eps_u == nullptr || out == nullptr) return DIT_ERR_INVALID_ARG;
  if (numel < 1 || numel > (1LL << 46)) return DIT_ERR_INVALID_ARG;
  if (!std::isfinite(w)) return DIT_ERR_INVALID_ARG;
  if (!aligned16(eps_c) || !aligned16(eps_u) || !aligned16(out)) return DIT_ERR_MISALIGNED;
  // out may be exactly eps_c or eps_u; any other overlap is an error.
  const size_t bytes = static_cast<size_t>(numel) * 4;
  if ((out != eps_c && ranges_overlap(out, bytes, eps_c, bytes)) ||
      (out != eps_u && ranges_overlap(out, bytes, eps_u, bytes)))
    return DIT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const long long n4 = numel / 4;
  if (n4 > 0) {
    if (launch_pdl(ditk::cfg_combine_vec4_kernel, dim3(stream_grid(*st, n4)), dim3(ditk::kStreamThreads), 0, cs,
                   reinterpret_cast<const float4 *>(eps_c), reinterpret_cast<const float4 *>(eps_u), w,
                   reinterpret_cast<float4 *>(out), n4) != cudaSuccess)
      return DIT_ERR_LAUNCH;
  }
  if (numel % 4 != 0) {
    if (launch_pdl(ditk::cfg_combine_tail_kernel, dim3(1), dim3(32), 0, cs, eps_c, eps_u, w, out, n4 * 4, numel) !=
        cudaSuccess)
      return DIT_ERR_LAUNCH;
  }
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status cfg_combine_relmae(const float *eps_c, const float *eps_u, float w, float *out, long long numel,
                              double *sums, dit_stream_t stream) {
  if (eps_c == nullptr || eps_u == nullptr || out == nullptr || sums == nullptr) return DIT_ERR_INVALID_ARG;
  if (numel < 1 || numel > (1LL << 46)) return DIT_ERR_INVALID_ARG;
  if (!std::isfinite(w)) return DIT_ERR_INVALID_ARG;
  if (!aligned16(eps_c) || !aligned16(eps_u) || !aligned16(out) || (reinterpret_cast<uintptr_t>(sums) & 7u) != 0)
    return DIT_ERR_MISALIGNED;
  // out may be exactly eps_c or eps_u; any other overlap is an error.
  const size_t bytes = static_cast<size_t>(numel) * 4;
  if ((out != eps_c && ranges_overlap(out, bytes, eps_c, bytes)) ||
      (out != eps_u && ranges_overlap(out, bytes, eps_u, bytes)) || ranges_overlap(sums, 24, eps_c, bytes) ||
      ranges_overlap(sums, 24, eps_u, bytes) || ranges_overlap(sums, 24, out, bytes))
    return DIT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(sums, 0, 3 * sizeof(double), cs) != cudaSuccess) return DIT_ERR_CUDA;
  const long long n4 = numel / 4;
  const int grid = stream_grid(*st, n4 > 0 ? n4 : 1);
  if (launch_pdl(ditk::cfg_combine_relmae_kernel, dim3(grid), dim3(ditk::kStreamThreads), 0, cs, eps_c, eps_u, w, out,
                 numel, sums) != cudaSuccess)
    return DIT_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status cfg_combine_relmae_static(const float *eps_c, const float *eps_u, float w, float *out, long long numel,
                                     double *sums, dit_stream_t stream) {
  static_assert(DIT_RELMAE_STATIC_MAX_NUMEL == ditk::kRelmaeMaxNumel, "header limit out of step");
  if (eps_c == nullptr || eps_u == nullptr || out == nullptr || sums == nullptr) return DIT_ERR_INVALID_ARG;
  if (numel < 1 || numel > ditk::kRelmaeMaxNumel) return DIT_ERR_INVALID_ARG;
  if (!std::isfinite(w)) return DIT_ERR_INVALID_ARG;
  if (!aligned16(eps_c) || !aligned16(eps_u) || !aligned16(out) || (reinterpret_cast<uintptr_t>(sums) & 7u) != 0)
    return DIT_ERR_MISALIGNED;
  const size_t bytes = static_cast<size_t>(numel) * 4;
  if ((out != eps_c && ranges_overlap(out, bytes, eps_c, bytes)) ||
      (out != eps_u && ranges_overlap(out, bytes, eps_u, bytes)) || ranges_overlap(sums, 24, eps_c, bytes) ||
      ranges_overlap(sums, 24, eps_u, bytes) || ranges_overlap(sums, 24, out, bytes))
    return DIT_ERR_INVALID_ARG;
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  double *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_relmae_scratch_ptr[dev] == nullptr) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, ditk::g_relmae_scratch) != cudaSuccess || p == nullptr) return DIT_ERR_CUDA;
      g_relmae_scratch_ptr[dev] = static_cast<double *>(p);
    }
    scratch = g_relmae_scratch_ptr[dev];
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The ticket counter must start at zero; the per-block slots are written
  // before they are read.
  if (cudaMemsetAsync(scratch + ditk::kRelmaeTicket, 0, sizeof(unsigned long long), cs) != cudaSuccess)
    return DIT_ERR_CUDA;
  const int grid = static_cast<int>((numel + ditk::kRelmaeSlab - 1) / ditk::kRelmaeSlab);
  ditk::cfg_combine_relmae_slab_kernel<<<grid, ditk::kStreamThreads, 0, cs>>>(eps_c, eps_u, w, out, numel, sums,
                                                                             scratch);
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status dit_selftest_bounded_wait(dit_stream_t stream) {
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  ditk::selftest_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH;
}

dit_status dit_last_device_status(dit_stream_t stream) {
  int dev = 0;
  DeviceState *st = nullptr;
  dit_status s = select_device(stream, &dev, &st);
  if (s != DIT_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_status_mu);
  // After the work queued on the stream: take the word (read and clear in one
  // atomic exchange on the device), then copy what was taken back.
  ditk::status_take_kernel<<<1, 1, 0, cs>>>();
  if (cudaGetLastError() != cudaSuccess) return DIT_ERR_LAUNCH;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbolAsync(&word, ditk::g_status_taken, sizeof(word), 0, cudaMemcpyDeviceToHost, cs) !=
      cudaSuccess)
    return DIT_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return DIT_ERR_CUDA;
  return word != 0u ? DIT_ERR_DEVICE_TIMEOUT : DIT_OK;
}

}  // extern "C"
