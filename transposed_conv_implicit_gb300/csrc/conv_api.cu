// Host side of libconvgb300: argument validation (the acceptance gates), tile
// planning, TMA tensor-map encoding, the filter-packing kernels and the C ABI
// declared in include/conv_gb300.h.
//
// Gates follow "dispatch_amd_4wave_conv2d" (Parameters and Args): input dtype
// fp8-e4m3 / bf16 / fp16, filter dtype = input dtype, output bf16 for fp8
// inputs else the input dtype, stride (1,1) or (2,2), dilation (1,1),
// symmetric padding (0,0)/(1,1)/(2,2), one group.  A failed gate returns
// CONV_ERR_NOT_SUPPORTED: there is no fallback path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>

#include "../../include/conv_gb300.h"
#include "../../include/conv_gb300_testing.h"
#include "conv_internal.h"

using namespace convgb300;

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;  // one second per wait
constexpr int kMaxFilterExtent = 32;
constexpr size_t kSmemLimit = 227 * 1024;

std::atomic<int> g_fault_mode{0};
std::atomic<unsigned long long> g_timeout_ns{0};

int elt_bytes(conv_dtype_t d) { return d == CONV_DTYPE_F8E4M3 ? 1 : 2; }

// Tuning overrides read from the environment (0 or unset = let the planner
// choose): CONV_TILE_M (128 or 256), CONV_TILE_N (a multiple of 16, <= 256),
// CONV_FILTER_RESIDENT (0 forbids keeping the filter in shared memory),
// CONV_MAX_STAGES (caps the operand ring), CONV_SRC_BUFS (1: one residual
// source buffer), CONV_PAIR (1/0: force CTA pairs on/off), CONV_WINDOW,
// CONV_ROWTAP, CONV_GATHER_STAGE and CONV_L2_PREFETCH (-1 disables that
// loader or feature), CONV_ROWTAP_BAND, CONV_STREAMK (1/0: force the
// stream-K schedule on where it applies / off), CONV_MMA_SPLIT (0: one MMA
// issuer for both 128-row halves), CONV_WAIT_HINT_NS.  Read once
// per process, on first use; conv_testing_reload_tuning() reads them again.
struct Tuning {
  int tile_m, tile_n, max_stages, src_bufs, window, rowtap, rowtap_band, gather_stage, l2_prefetch;
  int filter_resident;  // -1 when unset
  int pair;             // -1 when unset
  int streamk;          // -1 when unset
  int mma_split;        // 0 disables the second MMA issuer
  int rowtap_blocks;    // row-tap A stage: 1 = one channel block, 0 = the planner's choice
  uint32_t wait_hint_ns;
};

int env_int(const char* name) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : 0;
}

int env_int_or(const char* name, int unset) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : unset;
}

Tuning read_tuning() {
  Tuning t{};
  t.tile_m = env_int("CONV_TILE_M");
  t.tile_n = env_int("CONV_TILE_N");
  t.max_stages = env_int("CONV_MAX_STAGES");
  t.src_bufs = env_int("CONV_SRC_BUFS");
  t.window = env_int("CONV_WINDOW");
  t.rowtap = env_int("CONV_ROWTAP");
  t.rowtap_band = env_int("CONV_ROWTAP_BAND");
  t.gather_stage = env_int("CONV_GATHER_STAGE");
  t.l2_prefetch = env_int("CONV_L2_PREFETCH");
  t.filter_resident = env_int_or("CONV_FILTER_RESIDENT", -1);
  t.pair = env_int_or("CONV_PAIR", -1);
  t.streamk = env_int_or("CONV_STREAMK", -1);
  t.mma_split = env_int_or("CONV_MMA_SPLIT", 1);
  t.rowtap_blocks = env_int("CONV_ROWTAP_BLOCKS");
  t.wait_hint_ns = static_cast<uint32_t>(env_int("CONV_WAIT_HINT_NS"));
  return t;
}

std::mutex g_tuning_mu;
Tuning g_tuning_value;
std::atomic<unsigned> g_tuning_gen{0};  // 0: not read yet; bumped by every (re)load

const Tuning& tuning() {
  if (g_tuning_gen.load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lock(g_tuning_mu);
    if (g_tuning_gen.load(std::memory_order_relaxed) == 0) {
      g_tuning_value = read_tuning();
      g_tuning_gen.store(1, std::memory_order_release);
    }
  }
  return g_tuning_value;
}

bool known_dtype(conv_dtype_t d) {
  return d == CONV_DTYPE_BF16 || d == CONV_DTYPE_F16 || d == CONV_DTYPE_F8E4M3;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ driver
struct DriverFns {
  PFN_cuTensorMapEncodeIm2col_v12000 im2col = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 tiled = nullptr;
};

const DriverFns* driver_fns() {
  static DriverFns fns;
  static bool ok = false;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q1{}, q2{};
    void* p1 = nullptr;
    void* p2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p1, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p2, 12000, cudaEnableDefault,
                                         &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !p1 || !p2) {
      return;
    }
    fns.im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(p1);
    fns.tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p2);
    ok = true;
  });
  return ok ? &fns : nullptr;
}

// Cycles of the SM clock in `ns` nanoseconds (at the device's rated clock;
// a throttled clock only makes the bounded waits last longer).
long long ns_to_cycles(unsigned long long ns) {
  static std::atomic<int> khz_cache[64];
  int dev = 0;
  int khz = 2100000;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    int v = khz_cache[dev].load(std::memory_order_relaxed);
    if (v <= 0 && cudaDeviceGetAttribute(&v, cudaDevAttrClockRate, dev) == cudaSuccess && v > 0)
      khz_cache[dev].store(v, std::memory_order_relaxed);
    if (v > 0) khz = v;
  }
  return static_cast<long long>(ns / 1000ull) * khz / 1000ll + 1;
}

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

CUtensorMapDataType tmap_dtype(conv_dtype_t d) {
  if (d == CONV_DTYPE_BF16) return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (d == CONV_DTYPE_F16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // fp8 moves as raw bytes
}

CUtensorMapSwizzle tmap_swizzle(uint32_t row_bytes) {
  if (row_bytes == 128) return CU_TENSOR_MAP_SWIZZLE_128B;
  if (row_bytes == 64) return CU_TENSOR_MAP_SWIZZLE_64B;
  return CU_TENSOR_MAP_SWIZZLE_32B;
}

// ------------------------------------------------------------------ planning
struct Plan {
  ConvKernelParams kp;
  conv_dtype_t in_dtype;
  bool out_bf16;
  int kind;
  int phases_packed;   // phase slots in the packed filter
  int kmax;            // packed K per phase slot
  size_t packed_bytes;
  int grid;
  size_t smem_bytes;
  size_t sk_offset;    // stream-K flags and partial slots: this far into the workspace
};

// Channels per k-block: rows of 128, 64 or 32 bytes (the swizzle span).  The
// last block of a filter tap may reach past C_in: the TMA zero-fills those
// channels of A, so the filter values they meet (the next tap's, or zero
// fill past K) contribute nothing.  Prefer 128-byte rows unless that wastes
// more than a quarter of the MMA work; C_in * elt must be a multiple of 16
// bytes (TMA strides and coordinates) and at least 32 bytes (one MMA K-step).
conv_status_t channel_block(int c_in, int elt, int* bk, uint32_t* row_bytes) {
  const long long cb = static_cast<long long>(c_in) * elt;
  if (cb % 16 != 0 || cb < 32) return CONV_ERR_NOT_SUPPORTED;
  uint32_t rb = 32;
  if (cb % 128 == 0 || (cb > 128 && ((cb + 127) / 128) * 128 * 4 <= cb * 5)) {
    rb = 128;
  } else if (cb % 64 == 0 || (cb > 64 && ((cb + 63) / 64) * 64 * 4 <= cb * 5)) {
    rb = 64;
  }
  *row_bytes = rb;
  *bk = static_cast<int>(rb) / elt;
  return CONV_OK;
}

FastDiv make_fast_div(uint32_t d) {
  FastDiv f{};
  f.d = d;
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  f.shift = s;
  f.mul = static_cast<uint32_t>((((1ull << 32) * ((1ull << s) - d)) / d + 1) & 0xFFFFFFFFull);
  return f;
}

// Forward convs whose channel rows a TMA box cannot address (C_in * elt not
// a multiple of 16 bytes, or under 32) use the gather A loader.  Its
// contraction layout: per filter row r one run of S taps x C_in channels
// (S * C_in * elt bytes, contiguous in the NHWC input when dil_w = 1),
// zero-padded to a multiple of 16 bytes; the packed filter follows it.
bool gather_mode(int c_in, int elt) {
  const long long cb = static_cast<long long>(c_in) * elt;
  return cb % 16 != 0 || cb < 32;
}

uint32_t align1k(size_t v) { return static_cast<uint32_t>((v + 1023) & ~static_cast<size_t>(1023)); }

// Shared memory of the gather loader beyond the barriers: one row table per
// producer warp (16 bytes per tile row) and, when input rows are staged, two
// staging buffers.  Decides whether rows are staged (sets g_stage, g_slots,
// g_stage_bytes); needs m_halves.
size_t gather_smem_bytes(ConvKernelParams& kp) {
  if (!kp.gather) return 0;
  const size_t tables = static_cast<size_t>(kGatherProducers) * kBM * kp.m_halves * 16;
  kp.g_stage = 0;
  kp.g_slots = 0;
  kp.g_stage_bytes = 0;
  if (kp.g_row_bytes % 16 == 0 && tuning().gather_stage != -1) {
    // Padded rows a tile of `rows` consecutive output pixels can touch: its
    // output rows (at most (rows-1)/Wo + 2 of them) step stride_h apart, plus
    // the filter extent, plus, at each image boundary crossed, the rest of
    // the filter extent of the image it leaves.
    const long long rows = static_cast<long long>(kBM) * kp.m_halves;
    const long long out_rows = (rows - 1) / kp.Wo + 2;
    const long long ext = static_cast<long long>(kp.g_runs - 1) * kp.dil_h + 1;
    const long long crossings =
        std::min(out_rows - 1, (rows - 1) / (static_cast<long long>(kp.Ho) * kp.Wo) + 1);
    const long long slots = (out_rows - 1) * kp.step_h + ext +
                            crossings * std::max<long long>(0, ext - kp.step_h);
    // Zero margins: a piece may start pad_w pixels left of the row (minus the
    // 3 bytes of 4-byte rounding) and end pad_w pixels plus a run's padding
    // and the 20-byte read window right of it.
    const long long pix = kp.g_row_bytes / kp.g_w;
    const long long pad_l = ((-kp.base_w[0]) * pix + 4 + 15) / 16 * 16;
    const long long pad_r = ((-kp.base_w[0]) * pix + 32 + 15) / 16 * 16;
    const long long slot = pad_l + kp.g_row_bytes + pad_r;
    const size_t buf = align1k(static_cast<size_t>(slots * slot));
    if (2 * buf <= 96 * 1024) {
      kp.g_stage = 1;
      kp.g_slots = static_cast<int>(slots);
      kp.g_slot_bytes = static_cast<int>(slot);
      kp.g_slot_pad = static_cast<int>(pad_l);
      kp.g_stage_bytes = static_cast<uint32_t>(buf);
    }
  }
  return align1k(tables) + 2 * static_cast<size_t>(kp.g_stage_bytes);
}

// Grouped convs run on the tensor cores (TMA im2col loader) when a group's
// input channels are whole channel blocks of TMA rows, so that no load
// reaches into the next group; otherwise on the direct CUDA-core kernel.
bool groups_on_tensor_cores(int c_group, int elt) {
  int bk = 0;
  uint32_t rb = 0;
  return !gather_mode(c_group, elt) && channel_block(c_group, elt, &bk, &rb) == CONV_OK &&
         c_group % bk == 0;
}

long long gather_run_bytes(int s, int c_in, int elt) {
  return ((static_cast<long long>(s) * c_in * elt + 15) / 16) * 16;
}

// Packed K (elements per output channel) of the forward filter.
long long fwd_packed_k(int r, int s, int c_in, int elt) {
  if (gather_mode(c_in, elt)) return r * gather_run_bytes(s, c_in, elt) / elt;
  return static_cast<long long>(r) * s * c_in;
}

uint32_t make_idesc(conv_dtype_t in, int bn, int m = kBM) {
  // kind::f16: A/B format 0 = fp16, 1 = bf16; kind::f8f6f4: 0 = e4m3.
  // D format (bits 4-5) 1 = fp32; both operands K-major (bits 15, 16 = 0);
  // N >> 3 in bits 17-22; M >> 4 in bits 24-28.
  uint32_t fmt = in == CONV_DTYPE_BF16 ? 1u : 0u;
  uint32_t d = 0;
  d |= 1u << 4;
  d |= fmt << 7;
  d |= fmt << 10;
  d |= (static_cast<uint32_t>(bn) >> 3) << 17;
  d |= (static_cast<uint32_t>(m) >> 4) << 24;
  return d;
}

uint32_t next_pow2_cols(int cols) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(cols)) c <<= 1;
  return c;
}

conv_status_t encode_input_map(CUtensorMap* map, const void* input, int n, int h, int w, int c,
                               conv_dtype_t dt, int bk, uint32_t row_bytes, int pixels, int lower_w,
                               int lower_h, int upper_w, int upper_h, int step_w, int step_h) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  if (lower_w < -128 || lower_w > 127 || lower_h < -128 || lower_h > 127 || upper_w < -128 ||
      upper_w > 127 || upper_h < -128 || upper_h > 127)
    return CONV_ERR_NOT_SUPPORTED;
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(dt));
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(c), static_cast<cuuint64_t>(w),
                        static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
  int lower[2] = {lower_w, lower_h};
  int upper[2] = {upper_w, upper_h};
  cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(step_w), static_cast<cuuint32_t>(step_h), 1};
  CUresult r = fns->im2col(map, tmap_dtype(dt), 4, const_cast<void*>(input), dims, strides, lower,
                           upper, static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(pixels), estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, tmap_swizzle(row_bytes),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}

conv_status_t encode_filter_map(CUtensorMap* map, const void* packed, int kmax, int c_out,
                                int phases, conv_dtype_t dt, int bk, int bn, uint32_t row_bytes) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(dt));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kmax), static_cast<cuuint64_t>(c_out),
                        static_cast<cuuint64_t>(phases)};
  cuuint64_t strides[2] = {dims[0] * e, dims[0] * dims[1] * e};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(bn), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fns->tiled(map, tmap_dtype(dt), 3, const_cast<void*>(packed), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, tmap_swizzle(row_bytes),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}

bool dtype_pair_ok(conv_dtype_t in, conv_dtype_t out) {
  if (!known_dtype(in) || !known_dtype(out)) return false;
  return in == CONV_DTYPE_F8E4M3 ? out == CONV_DTYPE_BF16 : out == in;
}

// Channel block, dtype and instruction kind (shared by forward and transposed plans).
conv_status_t plan_channels(Plan* pl, conv_dtype_t in, int c_in) {
  int bk = 0;
  uint32_t row_bytes = 0;
  conv_status_t st = channel_block(c_in, elt_bytes(in), &bk, &row_bytes);
  if (st != CONV_OK) return st;
  ConvKernelParams& kp = pl->kp;
  kp.bk = bk;
  kp.c_blocks = (c_in + bk - 1) / bk;
  kp.c_tail = c_in - kp.c_blocks * bk;
  kp.c_in = c_in;
  kp.sw_bytes = row_bytes;
  pl->in_dtype = in;
  pl->out_bf16 = (in != CONV_DTYPE_F16);
  pl->kind = in == CONV_DTYPE_F8E4M3 ? kKindF8 : kKindF16;
  return CONV_OK;
}

// Tile shape: the C_out tile width bn (a multiple of 16, <= 256) and the tile
// height (128 rows, or 256 rows as two 128-row MMAs sharing each filter
// k-block when bn <= 128).  A cost model from measurements on this part picks
// the shape with the shortest makespan over the persistent grid:
//  - one tcgen05.mma (M=128) occupies the tensor pipe ~63 cycles for N <= 128
//    and proportionally longer above (127 cycles at N=256);
//  - operand loads stream at ~70 bytes per cycle per SM, plus ~40 cycles of
//    issue per TMA instruction;
//  - a k-block costs the larger of the two; a tile adds its epilogue.
void choose_tiling(Plan* pl, const long long rows[], int num_phases, int max_kblocks, int c_out,
                   int num_sms) {
  ConvKernelParams& kp = pl->kp;
  double best = 1e300;
  int best_bn = 16, best_nt = 1, best_mh = 1;
  const int nt_min = (c_out + 255) / 256;
  const int nt_max = std::max(nt_min, std::min((c_out + 15) / 16, nt_min + 8));
  const int ksteps = static_cast<int>(kp.sw_bytes / 32);
  for (int mh = 2; mh >= 1; --mh) {
    for (int nt = nt_min; nt <= nt_max; ++nt) {
      const int per = (c_out + nt - 1) / nt;
      const int bn = ((per + 15) / 16) * 16;
      if (bn > 256 || (mh == 2 && bn > 128)) continue;
      const int nte = (c_out + bn - 1) / bn;
      long long tiles = 0;
      for (int ph = 0; ph < num_phases; ++ph) tiles += ((rows[ph] + kBM * mh - 1) / (kBM * mh)) * nte;
      const long long waves = (tiles + num_sms - 1) / std::max(num_sms, 1);
      const double a = static_cast<double>(kBM) * mh * kp.sw_bytes;
      const double b = static_cast<double>(bn) * kp.sw_bytes;
      const bool res = num_phases == 1 && nte == 1 && max_kblocks * b <= 96.0 * 1024;
      // The gather loader builds A at ~11 cycles per row per warp, with three warps.
      const double load = kp.gather ? std::max(kBM * mh * 3.7, (res ? 0.0 : b) / 70.0 + 40.0)
                                    : (a + (res ? 0.0 : b)) / 70.0 + 40.0 * (res ? 1 : 2);
      const double mma = static_cast<double>(mh) * ksteps * (63.0 * std::max(1.0, bn / 128.0) + 8.0);
      const double epi = static_cast<double>(kBM) * mh * bn * 2 / 64.0;
      // The smaller term still costs a little (issue slots, barriers): it breaks
      // ties in favour of fewer, wider MMAs.
      // A gather tile also pays fixed work of ~2,000 cycles: each builder
      // warp's row table and the row-staging handshake (the RGB stem ran
      // 77.8 us on 256-row tiles against 90.1 on 128-row ones).
      const double tile = max_kblocks * (std::max(load, mma) + 0.1 * std::min(load, mma)) + epi +
                          (kp.gather ? 2000.0 : 0.0);
      const double cost = waves * tile;
      if (cost < best * 0.999) {
        best = cost;
        best_bn = bn;
        best_nt = nte;
        best_mh = mh;
      }
    }
  }
  const int force_m = tuning().tile_m;
  const int force_n = tuning().tile_n;
  if (force_n >= 16 && force_n <= 256 && force_n % 16 == 0) {
    best_bn = force_n;
    best_nt = (c_out + force_n - 1) / force_n;
    if (best_bn > 128) best_mh = 1;
  }
  if (force_m == 128) best_mh = 1;
  if (force_m == 256 && best_bn <= 128) best_mh = 2;
  kp.bn = best_bn;
  kp.n_tiles = best_nt;
  kp.m_halves = best_mh;
  kp.acc_stride = static_cast<uint32_t>(best_mh * best_bn);
  kp.tmem_cols = next_pow2_cols(2 * best_mh * best_bn);
  kp.idesc = make_idesc(pl->in_dtype, best_bn);
}

// CTA pairs (cta_group::2): a cluster of two CTAs shares each 256-row tile;
// each CTA loads its 128 rows of A and half of the tile's bn filter rows, so
// per SM the filter bytes written into shared memory halve (measured: the
// VAE 3x3 512->512 conv, bn = 256, 194.6 -> 181.3 us; the fp8 3x3 320->320
// conv, bn = 160, 64.5 -> 61.7 us).  The gain is that share of the
// shared-memory traffic, so the default takes pairs only for filter-heavy
// tiles (bn > 128: B more than the A bytes per k-block; 256-row tiles of
// bn = 128 ran 12-30% slower as pairs) and only when every pair gets at
// least 4 tiles (pairs halve the tile slots).  For the TMA im2col loader
// with a streamed filter and one channel group.  CONV_PAIR=1 forces pairs
// where they apply, 0 forbids them.
void plan_pair(Plan* pl, int num_sms) {
  ConvKernelParams& kp = pl->kp;
  kp.pair = 0;
  const int force = tuning().pair;
  if (force == 0) return;
  if (kp.window || kp.gather || kp.groups > 1 || kp.bn < 32) return;
  const int tile_m = 2 * kBM;
  int tile = 0;
  for (int ph = 0; ph < kp.num_phases; ++ph)
    tile += ((kp.rows[ph] + tile_m - 1) / tile_m) * kp.n_tiles;
  if (force != 1 && (kp.bn <= kBM || tile < 4 * std::max(num_sms / 2, 1))) return;
  kp.pair = 1;
  kp.m_halves = 1;
  tile = 0;
  for (int ph = 0; ph < kp.num_phases; ++ph) {
    kp.tile_start[ph] = tile;
    tile += ((kp.rows[ph] + tile_m - 1) / tile_m) * kp.n_tiles;
  }
  kp.tile_start[kp.num_phases] = tile;
  kp.total_tiles = tile;
  kp.tiles_per_group = tile;
  kp.acc_stride = static_cast<uint32_t>(kp.bn);
  kp.tmem_cols = next_pow2_cols(2 * kp.bn);
  kp.idesc = make_idesc(pl->in_dtype, kp.bn, 2 * kBM);
}

// Stream-K schedule: when the tiles fill less than one wave of CTAs, the
// sequence of (tile, k-block) iterations is cut into one equal share per SM
// (work items end at tile boundaries); a tile split between CTAs is summed
// through fp32 partial slots in the workspace.  Cost model, in k-block
// times: the tile-per-CTA schedule's k-blocks per tile against the even share
// plus the fix-up.  Measured on this part, writing a 128 KB partial tile and
// reading it back take ~8 us of a CTA's critical path, against ~0.47 us for
// a 48 KB k-block: the fix-up is charged as 8x the partial tile's bytes in
// k-block loads, so stream-K pays for few tiles with a long contraction
// (small images with many channels), not for the benchmark convs.
// Needs `room` workspace bytes (streamk_bytes); TMA im2col loader, streamed
// filter, no CTA pairs, one channel group, every phase with filter taps.
// CONV_STREAMK=1 forces it where it applies, 0 forbids it.
size_t sk_slot_bytes(const ConvKernelParams& kp) {
  return static_cast<size_t>(kBM) * kp.m_halves * kp.bn * sizeof(float);
}

size_t sk_flag_bytes(int ctas) {
  return (static_cast<size_t>(ctas) * kEpilogueWarps * sizeof(unsigned int) + 255) & ~size_t(255);
}

size_t streamk_bytes(const ConvKernelParams& kp, int ctas) {
  return sk_flag_bytes(ctas) + static_cast<size_t>(ctas) * sk_slot_bytes(kp);
}

void plan_streamk(Plan* pl, int num_sms, size_t room) {
  ConvKernelParams& kp = pl->kp;
  kp.streamk = 0;
  const int force = tuning().streamk;
  if (force == 0 || num_sms < 2) return;
  if (kp.pair || kp.window || kp.gather || kp.groups > 1) return;
  long long iters = 0;
  int kpt_max = 0;
  for (int ph = 0; ph < kp.num_phases; ++ph) {
    const int kpt = kp.taps_h[ph] * kp.taps_w[ph] * kp.c_blocks;
    if (kpt <= 0) return;
    kpt_max = std::max(kpt_max, kpt);
    iters += static_cast<long long>(kp.tile_start[ph + 1] - kp.tile_start[ph]) * kpt;
  }
  if (iters <= 0 || iters >= (1ll << 31)) return;
  if (room < streamk_bytes(kp, num_sms)) return;
  if (force != 1) {
    if (kp.total_tiles >= num_sms) return;  // a full wave or more: whole tiles
    const long long share = (iters + num_sms - 1) / num_sms;
    const double kblock_bytes = static_cast<double>(kBM * kp.m_halves + kp.bn) * kp.sw_bytes;
    const double fixup = 8.0 * static_cast<double>(sk_slot_bytes(kp)) / kblock_bytes;
    if (kpt_max < 4 || static_cast<double>(share) + fixup > 0.85 * kpt_max) return;
  }
  kp.streamk = 1;
  kp.sk_iters = iters;
  long long it = 0;
  for (int ph = 0; ph < kMaxPhases; ++ph) {
    kp.sk_iter_start[ph] = it;
    if (ph < kp.num_phases) {
      const int kpt = kp.taps_h[ph] * kp.taps_w[ph] * kp.c_blocks;
      kp.sk_kpt[ph] = kpt;
      kp.sk_div_kpt[ph] = make_fast_div(static_cast<uint32_t>(kpt));
      it += static_cast<long long>(kp.tile_start[ph + 1] - kp.tile_start[ph]) * kpt;
    } else {
      kp.sk_kpt[ph] = 1;
      kp.sk_div_kpt[ph] = make_fast_div(1u);
    }
  }
  kp.sk_iter_start[kMaxPhases] = it;
  kp.sk_slot_floats = static_cast<uint32_t>(sk_slot_bytes(kp) / sizeof(float));
  kp.l2_prefetch = 0;
}

struct FwdShape {
  int n, h, w, c_in, r, s, c_out, ho, wo;
  int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  int groups;  // channel groups (num_groups)
  conv_dtype_t in_dtype, out_dtype;
};

conv_status_t check_fwd_shape(const FwdShape& f, int num_groups) {
  if (f.n <= 0 || f.h <= 0 || f.w <= 0 || f.c_in <= 0 || f.r <= 0 || f.s <= 0 || f.c_out <= 0)
    return CONV_ERR_INVALID_VALUE;
  if (!known_dtype(f.in_dtype) || !known_dtype(f.out_dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (!dtype_pair_ok(f.in_dtype, f.out_dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (!((f.stride_h == 1 && f.stride_w == 1) || (f.stride_h == 2 && f.stride_w == 2)))
    return CONV_ERR_NOT_SUPPORTED;
  if (f.dil_h < 1 || f.dil_w < 1 || f.dil_h > kMaxFilterExtent || f.dil_w > kMaxFilterExtent)
    return CONV_ERR_NOT_SUPPORTED;
  // Padding per axis, up to the dilated filter extent minus one (beyond it
  // whole output rows would see only padding).
  if (f.pad_h < 0 || f.pad_w < 0 || f.pad_h > f.dil_h * (f.r - 1) || f.pad_w > f.dil_w * (f.s - 1))
    return CONV_ERR_NOT_SUPPORTED;
  if (num_groups < 1 || f.c_in % num_groups != 0 || f.c_out % num_groups != 0)
    return CONV_ERR_INVALID_VALUE;
  // Narrow channel groups run on the direct kernel, whose filter slice must
  // fit in shared memory.
  if (num_groups > 1 && !groups_on_tensor_cores(f.c_in / num_groups, elt_bytes(f.in_dtype)) &&
      direct_smem_bytes(f.r, f.s, f.c_in / num_groups) > 200 * 1024)
    return CONV_ERR_NOT_SUPPORTED;
  // The gather loader reads S adjacent pixels per filter row and indexes
  // input pixels with 32-bit integers.
  if (num_groups == 1 && gather_mode(f.c_in, elt_bytes(f.in_dtype)) &&
      (f.dil_w != 1 || static_cast<long long>(f.n) * f.h * f.w >= (1ll << 30)))
    return CONV_ERR_NOT_SUPPORTED;
  if (f.r > kMaxFilterExtent || f.s > kMaxFilterExtent) return CONV_ERR_NOT_SUPPORTED;
  const long long ho = (static_cast<long long>(f.h) + 2 * f.pad_h - f.dil_h * (f.r - 1) - 1) /
                           f.stride_h + 1;
  const long long wo = (static_cast<long long>(f.w) + 2 * f.pad_w - f.dil_w * (f.s - 1) - 1) /
                           f.stride_w + 1;
  if (f.h + 2 * f.pad_h < f.dil_h * (f.r - 1) + 1 || f.w + 2 * f.pad_w < f.dil_w * (f.s - 1) + 1)
    return CONV_ERR_INVALID_VALUE;
  if (ho != f.ho || wo != f.wo) return CONV_ERR_INVALID_VALUE;
  const long long rows = static_cast<long long>(f.n) * f.ho * f.wo;
  if (rows > (1ll << 30)) return CONV_ERR_NOT_SUPPORTED;
  return CONV_OK;
}


// Row-window A loader for stride-1 forward convs: when a padded output row
// (Wo + S - 1 pixels) fits in one 128-row MMA half, the tile's input rows are
// loaded once per channel block and every filter tap reads them at a row
// offset, instead of one im2col box per tap.  Needs 128-byte channel rows,
// 16-byte output rows and one resident C_out tile.  CONV_WINDOW=-1 disables.
conv_status_t layout_memory_window(Plan* pl, int has_residual);

void plan_window(const FwdShape& f, Plan* pl, int num_sms, int has_residual) {
  ConvKernelParams& kp = pl->kp;
  kp.window = 0;
  if (tuning().window == -1) return;
  if (f.stride_h != 1 || f.stride_w != 1 || f.dil_h != 1 || f.dil_w != 1) return;
  if (kp.sw_bytes != 128 || !kp.vec_ok) return;
  const int pitch = f.wo + f.s - 1;
  if (pitch > kBM || f.c_out > 256) return;
  const int bn = ((f.c_out + 15) / 16) * 16;
  const size_t bres = static_cast<size_t>(f.r) * f.s * kp.c_blocks * bn * kp.sw_bytes;
  if (bres > 120 * 1024) return;
  const int mh = bn <= 128 ? 2 : 1;
  const int rows = kBM / pitch;
  const int rows_tile = mh * rows;
  const int row_blocks = (f.ho + rows_tile - 1) / rows_tile;
  (void)num_sms;
  kp.window = 1;
  kp.bn = bn;
  kp.n_tiles = 1;
  kp.m_halves = mh;
  kp.acc_stride = static_cast<uint32_t>(mh * bn);
  kp.tmem_cols = next_pow2_cols(2 * mh * bn);
  kp.idesc = make_idesc(pl->in_dtype, bn);
  kp.win_pitch = pitch;
  kp.win_rows = rows;
  kp.win_half_rows = rows * pitch;
  kp.win_box_rows = rows_tile + f.r - 1;
  kp.win_row_blocks = row_blocks;
  kp.win_R = f.r;
  kp.win_S = f.s;
  kp.win_pad_h = f.pad_h;
  kp.win_pad_w = f.pad_w;
  // The last junk rows of the last half read past the box: cover them.
  const int last_row = (mh - 1) * kp.win_half_rows + (f.r - 1) * pitch + (f.s - 1) + kBM;
  const size_t rows_needed = std::max<size_t>(static_cast<size_t>(pitch) * kp.win_box_rows, last_row);
  kp.win_stage_bytes = align1k(rows_needed * kp.sw_bytes);
  kp.total_tiles = f.n * row_blocks;
  kp.tile_start[0] = 0;
  kp.tile_start[1] = kp.total_tiles;
}

// Tries the row-window plan; keeps the im2col plan if it does not fit.
void plan_window_or_keep(const FwdShape& f, Plan* pl, int num_sms, int has_residual) {
  const Plan saved = *pl;
  plan_window(f, pl, num_sms, has_residual);
  if (pl->kp.window && layout_memory_window(pl, has_residual) != CONV_OK) *pl = saved;
}

// The gather loader's k-blocks: 128-byte rows (64 bf16/f16 or 128 fp8
// elements) over the run layout; the last block reaches past K, where the
// builder writes zeros and the filter map zero-fills.
conv_status_t plan_gather(const FwdShape& f, Plan* pl) {
  ConvKernelParams& kp = pl->kp;
  const int elt = elt_bytes(f.in_dtype);
  const long long run_bytes = gather_run_bytes(f.s, f.c_in, elt);
  const long long kbytes = f.r * run_bytes;
  if (kbytes > (1ll << 24)) return CONV_ERR_NOT_SUPPORTED;
  kp.bk = 128 / elt;
  kp.sw_bytes = 128;
  kp.c_blocks = static_cast<int>((kbytes + 127) / 128);
  kp.c_tail = 0;
  kp.c_in = f.c_in;
  kp.gather = 1;
  kp.g_n = f.n;
  kp.g_h = f.h;
  kp.g_w = f.w;
  kp.g_c = f.c_in;
  kp.g_elt = elt;
  kp.g_runs = f.r;
  kp.g_s = f.s;
  kp.g_run_len_bytes = f.s * f.c_in * elt;
  kp.g_run_bytes = static_cast<int>(run_bytes);
  const long long row_bytes = static_cast<long long>(f.w) * f.c_in * elt;
  kp.g_row_bytes = row_bytes < (1ll << 30) ? static_cast<int>(row_bytes) : 1;  // 1: never staged
  kp.g_pr = (f.ho - 1) * f.stride_h + (f.r - 1) * f.dil_h + 1;
  kp.g_div_run = make_fast_div(static_cast<uint32_t>(run_bytes));
  kp.g_div_pr = make_fast_div(static_cast<uint32_t>(kp.g_pr));
  pl->in_dtype = f.in_dtype;
  pl->out_bf16 = (f.in_dtype != CONV_DTYPE_F16);
  pl->kind = f.in_dtype == CONV_DTYPE_F8E4M3 ? kKindF8 : kKindF16;
  return CONV_OK;
}

conv_status_t plan_fwd(const FwdShape& f, Plan* pl, int num_sms, int has_residual,
                       size_t sk_room = 0) {
  std::memset(pl, 0, sizeof(*pl));
  const int groups = std::max(f.groups, 1);
  const int cg = f.c_in / groups, fg = f.c_out / groups;
  const bool gather = gather_mode(cg, elt_bytes(f.in_dtype));
  if (gather && groups > 1) return CONV_ERR_NOT_SUPPORTED;
  conv_status_t st = gather ? plan_gather(f, pl) : plan_channels(pl, f.in_dtype, cg);
  if (st != CONV_OK) return st;
  ConvKernelParams& kp = pl->kp;
  if (groups > 1 && kp.c_tail != 0) return CONV_ERR_NOT_SUPPORTED;
  kp.groups = groups;
  kp.c_group = cg;
  kp.f_group = fg;
  kp.num_phases = 1;
  kp.grid_h[0] = f.ho;
  kp.grid_w[0] = f.wo;
  kp.rows[0] = f.n * f.ho * f.wo;
  kp.taps_h[0] = gather ? 1 : f.r;  // gather k-blocks span the whole contraction
  kp.taps_w[0] = gather ? 1 : f.s;
  kp.base_h[0] = -f.pad_h;
  kp.base_w[0] = -f.pad_w;
  kp.out_off_h[0] = 0;
  kp.out_off_w[0] = 0;
  kp.b_index[0] = 0;
  kp.step_h = f.stride_h;
  kp.step_w = f.stride_w;
  kp.out_step_h = 1;
  kp.out_step_w = 1;
  kp.dil_h = f.dil_h;
  kp.dil_w = f.dil_w;
  // (Groups repeat the tile grid: the model sees all groups' rows.)
  const long long rows[1] = {static_cast<long long>(kp.rows[0]) * groups};
  choose_tiling(pl, rows, 1, kp.taps_h[0] * kp.taps_w[0] * kp.c_blocks, fg, num_sms);
  const int tile_m = kBM * kp.m_halves;
  const int m_tiles = (kp.rows[0] + tile_m - 1) / tile_m;
  kp.tile_start[0] = 0;
  kp.tile_start[1] = m_tiles * kp.n_tiles;
  kp.tiles_per_group = kp.tile_start[1];
  kp.total_tiles = kp.tile_start[1] * groups;
  kp.Ho = f.ho;
  kp.Wo = f.wo;
  kp.Cout = f.c_out;
  kp.vec_ok = (f.c_out * 2) % 16 == 0 && (fg * 2) % 16 == 0;
  pl->phases_packed = 1;
  pl->kmax = static_cast<int>(fwd_packed_k(f.r, f.s, cg, elt_bytes(f.in_dtype)));
  pl->packed_bytes = static_cast<size_t>(f.c_out) * pl->kmax * elt_bytes(f.in_dtype);
  if (!gather && groups == 1) plan_window_or_keep(f, pl, num_sms, has_residual);
  plan_pair(pl, num_sms);
  plan_streamk(pl, num_sms, sk_room);
  return CONV_OK;
}

// Encodes the forward conv's input map (lower corner -pad, upper corner
// pad - (S-1)*dil, element strides = conv stride).
conv_status_t encode_window_input(const FwdShape& f, const void* input, Plan* pl) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  const ConvKernelParams& kp = pl->kp;
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(f.in_dtype));
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(f.c_in), static_cast<cuuint64_t>(f.w),
                        static_cast<cuuint64_t>(f.h), static_cast<cuuint64_t>(f.n)};
  cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kp.bk), static_cast<cuuint32_t>(kp.win_pitch),
                       static_cast<cuuint32_t>(kp.win_box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fns->tiled(&pl->kp.map_a[0], tmap_dtype(f.in_dtype), 4, const_cast<void*>(input),
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          tmap_swizzle(kp.sw_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}

conv_status_t encode_fwd_input(const FwdShape& f, const void* input, Plan* pl) {
  if (pl->kp.gather) {  // plain loads: the kernel needs only the base and the extent
    pl->kp.g_input = static_cast<const uint8_t*>(input);
    pl->kp.g_input_bytes = static_cast<long long>(f.n) * f.h * f.w * f.c_in * elt_bytes(f.in_dtype);
    return CONV_OK;
  }
  if (pl->kp.window) return encode_window_input(f, input, pl);
  return encode_input_map(&pl->kp.map_a[0], input, f.n, f.h, f.w, f.c_in, f.in_dtype, pl->kp.bk,
                          pl->kp.sw_bytes, kBM * pl->kp.m_halves, -f.pad_w, -f.pad_h, f.pad_w - (f.s - 1) * f.dil_w,
                          f.pad_h - (f.r - 1) * f.dil_h, f.stride_w, f.stride_h);
}

// Stride-phase decomposition of the transposed conv along one axis, with
// stride st and dilation dil ("conv_transposed_gpu", Args: stride, dilation).
// Input i, tap r lands on output o = st*i - pad + r*dil.  Output index
// o = st*j + a (phase a) therefore receives tap r only when
// r*dil = a + pad (mod st): with g = gcd(dil, st) these taps are
// r0, r0 + st/g, r0 + 2*st/g, ... (none when g does not divide a + pad), and
// tap r reads input i = j + (a + pad - r*dil)/st.  Listing the T taps in
// reverse, u = T-1-k for r = r0 + k*st/g, the input row is j + L + u*dil/g
// with L = (a + pad - r_last*dil)/st: each phase is a stride-1 correlation
// with T taps at dilation dil/g, over the input shifted by L.
struct AxisPhase {
  int r0, taps, lower, grid;
  int rstep;  // st / g: filter index between consecutive taps of a phase
  int dil;    // dil / g: input index between consecutive taps
};

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

AxisPhase axis_phase(int a, int st, int pad, int R, int out_extent, int dil) {
  AxisPhase ph{};
  const int g = gcd_int(dil, st);
  ph.rstep = st / g;
  ph.dil = dil / g;
  ph.r0 = -1;
  for (int r = 0; r < std::min(R, ph.rstep) && ph.r0 < 0; ++r)
    if (((r * dil - a - pad) % st + st) % st == 0) ph.r0 = r;
  ph.taps = ph.r0 < 0 ? 0 : (R - ph.r0 + ph.rstep - 1) / ph.rstep;
  if (ph.taps > 0) {
    const int r_last = ph.r0 + (ph.taps - 1) * ph.rstep;
    ph.lower = (a + pad - r_last * dil) / st;  // exact: a + pad - r*dil is a multiple of st
  } else {
    ph.r0 = 0;
    ph.lower = 0;
  }
  ph.grid = out_extent > a ? (out_extent - a + st - 1) / st : 0;
  return ph;
}

// The packed transposed filter: one [C_out][kmax] K-major matrix per phase
// slot (slot = a * stride_w + b), phase (a, b) holding its taps in the order
// the kernel walks them.  Depends on filter extent, stride, dilation and
// padding only.
constexpr int kMaxTrSlots = 16;  // stride_h * stride_w phases at most
constexpr int kMaxTrLaunches = kMaxTrSlots / kMaxPhases;

struct TrPacking {
  int slots, kmax, sh, sw, rsh, rsw;
  int r0h[kMaxTrSlots], r0w[kMaxTrSlots], th[kMaxTrSlots], tw[kMaxTrSlots];
};

bool tr_packing(int r, int s, int c_in, const int stride[2], const int dilation[2],
                const int padding[2], TrPacking* pk) {
  std::memset(pk, 0, sizeof(*pk));
  if (stride[0] < 1 || stride[1] < 1 || stride[0] * stride[1] > kMaxTrSlots) return false;
  if (dilation[0] < 1 || dilation[1] < 1 || padding[0] < 0 || padding[1] < 0) return false;
  pk->slots = stride[0] * stride[1];
  pk->sh = stride[0];
  pk->sw = stride[1];
  int kmax = 0;
  for (int a = 0; a < stride[0]; ++a) {
    const AxisPhase ya = axis_phase(a, stride[0], padding[0], r, stride[0], dilation[0]);
    pk->rsh = ya.rstep;
    for (int b = 0; b < stride[1]; ++b) {
      const AxisPhase xb = axis_phase(b, stride[1], padding[1], s, stride[1], dilation[1]);
      pk->rsw = xb.rstep;
      const int slot = a * stride[1] + b;
      pk->r0h[slot] = ya.r0;
      pk->r0w[slot] = xb.r0;
      pk->th[slot] = ya.taps;
      pk->tw[slot] = xb.taps;
      kmax = std::max(kmax, ya.taps * xb.taps * c_in);
    }
  }
  pk->kmax = kmax ? kmax : c_in;  // keep the filter map well-formed
  return true;
}

struct TrShape {
  int n, h, w, c_in, r, s, c_out, ho, wo;
  int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  conv_dtype_t in_dtype, out_dtype;
};

// Gates of the transposed conv: strides up to kMaxTrSlots phases in all,
// dilation 1..32, 0 <= pad <= dil*(R-1), and the output size
// (h-1)*stride - 2*pad + dil*(R-1) + 1 plus an output padding in [0, stride).
conv_status_t check_tr_shape(const TrShape& t) {
  if (t.n <= 0 || t.h <= 0 || t.w <= 0 || t.c_in <= 0 || t.r <= 0 || t.s <= 0 || t.c_out <= 0 ||
      t.ho <= 0 || t.wo <= 0)
    return CONV_ERR_INVALID_VALUE;
  if (!known_dtype(t.in_dtype) || !known_dtype(t.out_dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (!dtype_pair_ok(t.in_dtype, t.out_dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (t.stride_h < 1 || t.stride_w < 1 || t.stride_h * t.stride_w > kMaxTrSlots)
    return CONV_ERR_NOT_SUPPORTED;
  if (t.dil_h < 1 || t.dil_w < 1 || t.dil_h > kMaxFilterExtent || t.dil_w > kMaxFilterExtent)
    return CONV_ERR_NOT_SUPPORTED;
  if (t.r > kMaxFilterExtent || t.s > kMaxFilterExtent) return CONV_ERR_NOT_SUPPORTED;
  if (t.pad_h < 0 || t.pad_w < 0 || t.pad_h > t.dil_h * (t.r - 1) || t.pad_w > t.dil_w * (t.s - 1))
    return CONV_ERR_NOT_SUPPORTED;
  const long long base_h =
      static_cast<long long>(t.h - 1) * t.stride_h - 2 * t.pad_h + t.dil_h * (t.r - 1) + 1;
  const long long base_w =
      static_cast<long long>(t.w - 1) * t.stride_w - 2 * t.pad_w + t.dil_w * (t.s - 1) + 1;
  if (t.ho - base_h < 0 || t.ho - base_h >= t.stride_h) return CONV_ERR_INVALID_VALUE;
  if (t.wo - base_w < 0 || t.wo - base_w >= t.stride_w) return CONV_ERR_INVALID_VALUE;
  const long long rows = static_cast<long long>(t.n) * t.ho * t.wo;
  if (rows > (1ll << 30)) return CONV_ERR_NOT_SUPPORTED;
  return CONV_OK;
}

// The phase slots of a transposed conv that have output pixels, in slot order.
int tr_active_slots(const TrShape& t, int out[kMaxTrSlots]) {
  int n = 0;
  for (int a = 0; a < t.stride_h; ++a) {
    const AxisPhase ya = axis_phase(a, t.stride_h, t.pad_h, t.r, t.ho, t.dil_h);
    for (int b = 0; b < t.stride_w; ++b) {
      const AxisPhase xb = axis_phase(b, t.stride_w, t.pad_w, t.s, t.wo, t.dil_w);
      if (ya.grid > 0 && xb.grid > 0) out[n++] = a * t.stride_w + b;
    }
  }
  return n;
}

// Plans one launch over the phase slots slots[0 .. nslots) (at most
// kMaxPhases): each is a dense stride-1 implicit GEMM over the input.
conv_status_t plan_transposed(const TrShape& t, const TrPacking& pk, const int* slots, int nslots,
                              Plan* pl, int num_sms, size_t sk_room = 0) {
  std::memset(pl, 0, sizeof(*pl));
  if (nslots < 1 || nslots > kMaxPhases) return CONV_ERR_INVALID_VALUE;
  conv_status_t st = plan_channels(pl, t.in_dtype, t.c_in);
  if (st != CONV_OK) return st;
  ConvKernelParams& kp = pl->kp;
  pl->phases_packed = pk.slots;
  int dil_h = 1, dil_w = 1;
  for (int ph = 0; ph < nslots; ++ph) {
    const int slot = slots[ph];
    const int a = slot / t.stride_w, b = slot - (slot / t.stride_w) * t.stride_w;
    const AxisPhase ya = axis_phase(a, t.stride_h, t.pad_h, t.r, t.ho, t.dil_h);
    const AxisPhase xb = axis_phase(b, t.stride_w, t.pad_w, t.s, t.wo, t.dil_w);
    dil_h = ya.dil;
    dil_w = xb.dil;
    kp.grid_h[ph] = ya.grid;
    kp.grid_w[ph] = xb.grid;
    kp.rows[ph] = t.n * ya.grid * xb.grid;
    // A phase without taps still runs (kblocks = 0): it writes act(0 + beta*source).
    kp.taps_h[ph] = ya.taps;
    kp.taps_w[ph] = xb.taps;
    kp.base_h[ph] = ya.lower;
    kp.base_w[ph] = xb.lower;
    kp.out_off_h[ph] = a;
    kp.out_off_w[ph] = b;
    kp.b_index[ph] = slot;
  }
  long long rows[kMaxPhases];
  int max_kb = 0;
  for (int ph = 0; ph < nslots; ++ph) {
    rows[ph] = kp.rows[ph];
    max_kb = std::max(max_kb, kp.taps_h[ph] * kp.taps_w[ph] * kp.c_blocks);
  }
  kp.num_phases = nslots;
  choose_tiling(pl, rows, nslots, max_kb, t.c_out, num_sms);
  const int tile_m = kBM * kp.m_halves;
  int tile = 0;
  for (int ph = 0; ph < nslots; ++ph) {
    kp.tile_start[ph] = tile;
    tile += ((kp.rows[ph] + tile_m - 1) / tile_m) * kp.n_tiles;
  }
  kp.tile_start[nslots] = tile;
  kp.total_tiles = tile;
  kp.step_h = 1;
  kp.step_w = 1;
  kp.out_step_h = t.stride_h;
  kp.out_step_w = t.stride_w;
  kp.dil_h = dil_h;  // the same for every phase of an axis
  kp.dil_w = dil_w;
  kp.Ho = t.ho;
  kp.Wo = t.wo;
  kp.Cout = t.c_out;
  kp.vec_ok = (t.c_out * 2) % 16 == 0;
  plan_pair(pl, num_sms);
  plan_streamk(pl, num_sms, sk_room);
  pl->kmax = pk.kmax;
  pl->packed_bytes = static_cast<size_t>(pk.slots) * t.c_out * pk.kmax * elt_bytes(t.in_dtype);
  return CONV_OK;
}

conv_status_t encode_tr_inputs(const TrShape& t, const void* input, Plan* pl) {
  ConvKernelParams& kp = pl->kp;
  for (int ph = 0; ph < kp.num_phases; ++ph) {
    // Base pixels walk grid_w x grid_h positions at step 1: upper corner so the
    // bounding box [lower, W-1+upper] holds exactly that many.
    const int upper_w = kp.grid_w[ph] - t.w + kp.base_w[ph];
    const int upper_h = kp.grid_h[ph] - t.h + kp.base_h[ph];
    conv_status_t st = encode_input_map(&kp.map_a[ph], input, t.n, t.h, t.w, t.c_in, t.in_dtype,
                                        kp.bk, kp.sw_bytes, kBM * kp.m_halves, kp.base_w[ph],
                                        kp.base_h[ph], upper_w,
                                        upper_h, 1, 1);
    if (st != CONV_OK) return st;
  }
  return CONV_OK;
}

// ------------------------------------------------------------------ packing kernels
template <typename T>
__global__ void pack_fwd_kernel(const T* __restrict__ w, T* __restrict__ out, int R, int S, int C,
                                int F, int fcrs) {
  const long long K = static_cast<long long>(R) * S * C;
  const long long total = K * F;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long f = idx / K;
    const long long k = idx - f * K;
    const long long c = k % C;
    const long long rs = k / C;
    const long long s = rs % S;
    const long long r = rs / S;
    out[idx] = fcrs ? w[((f * C + c) * R + r) * S + s] : w[((r * S + s) * C + c) * F + f];
  }
}

// Gather layout: out[f][r][j], j < run_elems, holds W(r, s, c, f) for
// j = s*C + c < S*C and zero in the run's padding.
template <typename T>
__global__ void pack_fwd_gather_kernel(const T* __restrict__ w, T* __restrict__ out, int R, int S,
                                       int C, int F, int fcrs, int run_elems) {
  const long long per_f = static_cast<long long>(R) * run_elems;
  const long long total = per_f * F;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long f = idx / per_f;
    const long long k = idx - f * per_f;
    const long long r = k / run_elems;
    const long long j = k - r * run_elems;
    T v = T(0);
    if (j < static_cast<long long>(S) * C) {
      const long long s = j / C;
      const long long c = j - s * C;
      v = fcrs ? w[((f * C + c) * R + r) * S + s] : w[((r * S + s) * C + c) * F + f];
    }
    out[idx] = v;
  }
}

template <typename T>
__global__ void pack_transposed_kernel(const T* __restrict__ w, T* __restrict__ out, int R, int S,
                                       int C, int F, TrPacking d) {
  const long long per_slot = static_cast<long long>(F) * d.kmax;
  const long long total = per_slot * d.slots;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int slot = static_cast<int>(idx / per_slot);
    const long long rem = idx - slot * per_slot;
    const long long f = rem / d.kmax;
    const long long k = rem - f * d.kmax;
    const long long tap = k / C;
    const long long c = k - tap * C;
    const int th = d.th[slot], tw = d.tw[slot];
    T v = T(0);
    if (tap < static_cast<long long>(th) * tw) {
      // Tap (uh, uw) of the phase: filter index r0 + rstep*(T-1-u) per axis.
      const int uh = static_cast<int>(tap / tw);
      const int uw = static_cast<int>(tap - static_cast<long long>(uh) * tw);
      const long long r = d.r0h[slot] + static_cast<long long>(d.rsh) * (th - 1 - uh);
      const long long s = d.r0w[slot] + static_cast<long long>(d.rsw) * (tw - 1 - uw);
      v = w[((r * S + s) * F + f) * C + c];  // RSFC [R][S][F][C]
    }
    out[idx] = v;
  }
}

int pack_grid(long long total) {
  long long blocks = (total + 255) / 256;
  return static_cast<int>(std::min<long long>(std::max<long long>(blocks, 1), 4096));
}

conv_status_t launch_pack_fwd(const void* filter, int r, int s, int c_in, int c_out, int fcrs,
                              conv_dtype_t dt, void* packed, cudaStream_t stream) {
  const int elt = elt_bytes(dt);
  if (gather_mode(c_in, elt)) {
    const int run_elems = static_cast<int>(gather_run_bytes(s, c_in, elt) / elt);
    const long long total = static_cast<long long>(r) * run_elems * c_out;
    if (elt == 2)
      pack_fwd_gather_kernel<uint16_t><<<pack_grid(total), 256, 0, stream>>>(
          static_cast<const uint16_t*>(filter), static_cast<uint16_t*>(packed), r, s, c_in, c_out,
          fcrs, run_elems);
    else
      pack_fwd_gather_kernel<uint8_t><<<pack_grid(total), 256, 0, stream>>>(
          static_cast<const uint8_t*>(filter), static_cast<uint8_t*>(packed), r, s, c_in, c_out,
          fcrs, run_elems);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
  }
  const long long total = static_cast<long long>(r) * s * c_in * c_out;
  if (elt_bytes(dt) == 2)
    pack_fwd_kernel<uint16_t><<<pack_grid(total), 256, 0, stream>>>(
        static_cast<const uint16_t*>(filter), static_cast<uint16_t*>(packed), r, s, c_in, c_out,
        fcrs);
  else
    pack_fwd_kernel<uint8_t><<<pack_grid(total), 256, 0, stream>>>(
        static_cast<const uint8_t*>(filter), static_cast<uint8_t*>(packed), r, s, c_in, c_out,
        fcrs);
  return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

conv_status_t launch_pack_tr(const TrPacking& d, const void* filter, int r, int s, int c_in,
                             int c_out, conv_dtype_t dt, void* packed, cudaStream_t stream) {
  const long long total = static_cast<long long>(d.slots) * c_out * d.kmax;
  if (elt_bytes(dt) == 2)
    pack_transposed_kernel<uint16_t><<<pack_grid(total), 256, 0, stream>>>(
        static_cast<const uint16_t*>(filter), static_cast<uint16_t*>(packed), r, s, c_in, c_out, d);
  else
    pack_transposed_kernel<uint8_t><<<pack_grid(total), 256, 0, stream>>>(
        static_cast<const uint8_t*>(filter), static_cast<uint8_t*>(packed), r, s, c_in, c_out, d);
  return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

// ------------------------------------------------------------------ epilogue + shared memory
conv_status_t plan_memory_direct(Plan* pl);

// The output (or source) as [rows][groups][c_out / groups]: a store box of cw
// channels x 1 group x 128 rows clips at the group's last channel as well as
// at the last row (groups = 1 is the plain [rows][c_out] matrix).
conv_status_t encode_out_map_grouped(CUtensorMap* map, const void* base, int c_out, int groups,
                                     long long rows, conv_dtype_t out_dt, int cw) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  const int fg = c_out / groups;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(fg), static_cast<cuuint64_t>(groups),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(fg) * 2, static_cast<cuuint64_t>(c_out) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(cw), 1, static_cast<cuuint32_t>(kBM)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fns->tiled(map, tmap_dtype(out_dt), 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, tmap_swizzle(cw * 2),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}

// The pixels of one stride phase of the output, as a 4-D tensor
// [N][grid_h][grid_w][C_out] with strides that skip the other phases.
conv_status_t encode_out_map_phase(CUtensorMap* map, const void* out, const ConvKernelParams& kp,
                                   int ph, int n, conv_dtype_t out_dt, int cw) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  const cuuint64_t e = 2, C = static_cast<cuuint64_t>(kp.Cout);
  const uint8_t* base = static_cast<const uint8_t*>(out) +
                        (static_cast<size_t>(kp.out_off_h[ph]) * kp.Wo + kp.out_off_w[ph]) * C * e;
  cuuint64_t dims[4] = {C, static_cast<cuuint64_t>(kp.grid_w[ph]),
                        static_cast<cuuint64_t>(kp.grid_h[ph]), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kp.out_step_w) * C * e,
                           static_cast<cuuint64_t>(kp.out_step_h) * kp.Wo * C * e,
                           static_cast<cuuint64_t>(kp.Ho) * kp.Wo * C * e};
  const int bw = kp.grid_w[ph] < kBM ? kp.grid_w[ph] : kBM;
  cuuint32_t box[4] = {static_cast<cuuint32_t>(cw), static_cast<cuuint32_t>(bw),
                       static_cast<cuuint32_t>(kBM / bw), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fns->tiled(map, tmap_dtype(out_dt), 4, const_cast<uint8_t*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, tmap_swizzle(cw * 2),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}


// Picks the epilogue mode, the filter residency and the ring depth so that
// everything fits in shared memory, and lays the buffers out.  No driver
// calls: the TMA maps of the epilogue are encoded afterwards.
conv_status_t layout_memory_window(Plan* pl, int has_residual);

conv_status_t layout_memory(Plan* pl, int has_residual) {
  ConvKernelParams& kp = pl->kp;
  if (kp.window) return layout_memory_window(pl, has_residual);
  // Epilogue mode: TMA tiles need 16-byte output rows; the transposed phase
  // grids additionally need every 128-row tile to be a rectangle of one image.
  int mode = 0;
  if (kp.vec_ok) {
    if (kp.num_phases == 1 && kp.out_step_h == 1 && kp.out_step_w == 1) {
      mode = 1;
    } else {
      mode = 2;
      for (int ph = 0; ph < kp.num_phases; ++ph) {
        const int gw = kp.grid_w[ph], gh = kp.grid_h[ph];
        const bool rect = (gw % kBM == 0) || (kBM % gw == 0 && gh % (kBM / gw) == 0);
        if (!rect) mode = 0;
      }
    }
  }
  if (mode == 0) return plan_memory_direct(pl);
  int cw = 16;
  for (int c : {64, 32, 16})
    if (kp.bn % c == 0) {
      cw = c;
      break;
    }
  // Two epilogue warpgroups split a tile's (half, chunk) items: make at least two.
  if (kp.m_halves * (kp.bn / cw) < kEpilogueGroups && cw > 16) cw /= 2;
  const uint32_t a_bytes = kBM * kp.m_halves * kp.sw_bytes;
  // (A pair's CTA holds half of the tile's filter rows.)
  const uint32_t b_bytes = static_cast<uint32_t>(kp.pair ? kp.bn / 2 : kp.bn) * kp.sw_bytes;
  const bool can_res = !kp.pair && !kp.streamk && kp.num_phases == 1 && kp.n_tiles == 1 &&
                       kp.groups <= 1 && tuning().filter_resident != 0;
  const size_t bres = can_res ? static_cast<size_t>(kp.taps_h[0]) * kp.taps_w[0] * kp.c_blocks * b_bytes : 0;
  const size_t src_tile = static_cast<size_t>(kBM) * kp.m_halves * kp.bn * 2;
  const size_t chunk = static_cast<size_t>(kBM) * cw * 2;
  const size_t bar_bytes = 1024 + gather_smem_bytes(kp);
  struct Opt { bool res; int srcb, stgb; };
  Opt opts[12];
  int nopt = 0;
  // CONV_SRC_BUFS (1 or 2) caps the residual-source tile buffers (tuning override).
  const int srcb_env = tuning().src_bufs;
  const int srcb_max = has_residual ? ((srcb_env == 1) ? 1 : 2) : 0;
  // With a residual the outputs are written in place into the source tile
  // buffer and stored from there: no staging buffers.
  const int stg_max = has_residual ? 0 : 2;
  const int stg_min = has_residual ? 0 : 1;
  for (int res = can_res ? 1 : 0; res >= 0; --res)
    for (int srcb = srcb_max; srcb >= (srcb_max ? 1 : 0); --srcb)
      for (int stgb = stg_max; stgb >= stg_min; --stgb) opts[nopt++] = Opt{res != 0, srcb, stgb};
  // Rank the options: at least 3 ring stages; then the cheapest k-block
  // (a resident filter saves one TMA load per k-block); then at least 5
  // stages; then a prefetched residual source; then deeper rings.
  int best = -1, best_stages = 0;
  double best_key = 1e300;
  for (int i = 0; i < nopt; ++i) {
    const size_t used = 1024 + bar_bytes + (opts[i].res ? align1k(bres) : 0) +
                        opts[i].srcb * align1k(src_tile) +
                        kEpilogueGroups * opts[i].stgb * align1k(chunk);
    const size_t stage = a_bytes + (opts[i].res ? 0 : b_bytes);
    if (used + 2 * stage > kSmemLimit) continue;
    int st = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - used) / stage));
    if (tuning().max_stages >= 2) st = std::min(st, tuning().max_stages);
    const double load = (a_bytes + (opts[i].res ? 0.0 : b_bytes)) / 70.0 + 40.0 * (opts[i].res ? 1 : 2);
    double key = load;
    if (st < 3) key += 1e6;
    if (opts[i].srcb < srcb_max) key += 50.0;
    // Below 6 stages a deeper ring beats the second source buffer (fp8 3x3
    // 320->320 with a residual: 4 stages and two source buffers 75.8 us
    // against 5 stages and one 73.7 us; on CTA pairs 5 stages and two
    // buffers 60.8 us against 7 stages and one 59.3 us).
    if (st < 6) key += 60.0;
    key -= 0.01 * st;
    if (key < best_key) {
      best_key = key;
      best = i;
      best_stages = st;
    }
  }
  if (best < 0) return plan_memory_direct(pl);
  const Opt o = opts[best];
  kp.epi_mode = mode;
  kp.cw = cw;
  kp.b_resident = o.res ? 1 : 0;
  kp.src_bufs = o.srcb;
  kp.src_chunk_bytes = static_cast<uint32_t>(chunk);
  kp.valid_rows = kBM;
  kp.stg_bufs = o.stgb;
  kp.stages = best_stages;
  uint32_t off = 0;
  kp.off_a = off;
  off += align1k(static_cast<size_t>(best_stages) * a_bytes);
  kp.off_b = off;
  if (!o.res) off += align1k(static_cast<size_t>(best_stages) * b_bytes);
  kp.off_bres = off;
  if (o.res) off += align1k(bres);
  kp.off_src = off;
  off += o.srcb * align1k(src_tile);
  kp.off_stg = off;
  off += kEpilogueGroups * o.stgb * align1k(chunk);
  kp.off_bar = off;
  kp.off_gtab = off + 1024;
  kp.off_gstage = kp.off_gtab + align1k(static_cast<size_t>(kGatherProducers) * kBM * kp.m_halves * 16);
  off += bar_bytes;
  pl->smem_bytes = off + 1024;
  return CONV_OK;
}

// Row-window mode: the resident filter, an A ring of whole-tile boxes (at
// least two), the residual-source tiles or output staging.
conv_status_t layout_memory_window(Plan* pl, int has_residual) {
  ConvKernelParams& kp = pl->kp;
  int cw = 16;
  for (int c : {64, 32, 16})
    if (kp.bn % c == 0) {
      cw = c;
      break;
    }
  if (kp.m_halves * (kp.bn / cw) < kEpilogueGroups && cw > 16) cw /= 2;
  const uint32_t b_bytes = static_cast<uint32_t>(kp.bn) * kp.sw_bytes;
  const size_t bres = static_cast<size_t>(kp.win_R) * kp.win_S * kp.c_blocks * b_bytes;
  // A source chunk holds only the half's stored rows (win_half_rows of 128).
  const size_t src_chunk = align1k(static_cast<size_t>(kp.win_half_rows) * cw * 2);
  const size_t src_tile = src_chunk * kp.m_halves * (kp.bn / cw);
  const size_t chunk = static_cast<size_t>(kBM) * cw * 2;
  const size_t bar_bytes = 1024;
  const size_t stage = kp.win_stage_bytes;
  int best_srcb = -1, best_stgb = -1, best_st = 0;
  for (int srcb = has_residual ? 2 : 0; srcb >= (has_residual ? 1 : 0); --srcb)
    for (int stgb = has_residual ? 0 : 2; stgb >= (has_residual ? 0 : 1); --stgb) {
      const size_t used = 1024 + bar_bytes + align1k(bres) + srcb * align1k(src_tile) +
                          kEpilogueGroups * stgb * align1k(chunk);
      if (used + 2 * stage > kSmemLimit) continue;
      int st = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - used) / stage));
      if (tuning().max_stages >= 2) st = std::min(st, tuning().max_stages);
      if (st > best_st) {
        best_st = st;
        best_srcb = srcb;
        best_stgb = stgb;
      }
    }
  if (best_st < 2) {  // does not fit: plain im2col tiles
    kp.window = 0;
    return CONV_ERR_NOT_SUPPORTED;
  }
  kp.epi_mode = 3;
  kp.cw = cw;
  kp.b_resident = 1;
  kp.src_bufs = best_srcb;
  kp.src_chunk_bytes = static_cast<uint32_t>(src_chunk);
  kp.valid_rows = kp.win_half_rows;
  kp.stg_bufs = best_stgb;
  kp.stages = best_st;
  uint32_t off = 0;
  kp.off_a = off;
  off += align1k(static_cast<size_t>(best_st) * stage);
  kp.off_b = off;
  kp.off_bres = off;
  off += align1k(bres);
  kp.off_src = off;
  off += best_srcb * align1k(src_tile);
  kp.off_stg = off;
  off += kEpilogueGroups * best_stgb * align1k(chunk);
  kp.off_bar = off;
  off += bar_bytes;
  pl->smem_bytes = off + 1024;
  return CONV_OK;
}

conv_status_t encode_out_map_window(CUtensorMap* map, const void* base, const ConvKernelParams& kp,
                                    int n, conv_dtype_t out_dt) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  const cuuint64_t e = 2, C = static_cast<cuuint64_t>(kp.Cout);
  cuuint64_t dims[4] = {C, static_cast<cuuint64_t>(kp.Wo), static_cast<cuuint64_t>(kp.Ho),
                        static_cast<cuuint64_t>(n)};
  cuuint64_t strides[3] = {C * e, C * e * kp.Wo, C * e * kp.Wo * kp.Ho};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kp.cw), static_cast<cuuint32_t>(kp.win_pitch),
                       static_cast<cuuint32_t>(kp.win_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fns->tiled(map, tmap_dtype(out_dt), 4, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, tmap_swizzle(kp.cw * 2),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV_OK : CONV_ERR_CUDA;
}

// Encodes the epilogue's output / source maps; falls back to the direct
// epilogue if the driver rejects one of them.
conv_status_t plan_memory(Plan* pl, int n_images, const void* output, const void* source,
                          int has_residual) {
  conv_status_t st = layout_memory(pl, has_residual);
  if (st != CONV_OK) return st;
  ConvKernelParams& kp = pl->kp;
  const conv_dtype_t out_dt = pl->out_bf16 ? CONV_DTYPE_BF16 : CONV_DTYPE_F16;
  if (kp.epi_mode == 3) {
    if (encode_out_map_window(&kp.map_out[0], output, kp, n_images, out_dt) != CONV_OK ||
        (has_residual &&
         encode_out_map_window(&kp.map_src[0], source, kp, n_images, out_dt) != CONV_OK))
      return CONV_ERR_CUDA;
  } else if (kp.epi_mode == 1) {
    const long long rows = kp.rows[0];
    if (encode_out_map_grouped(&kp.map_out[0], output, kp.Cout, kp.groups, rows, out_dt, kp.cw) !=
            CONV_OK ||
        (has_residual && encode_out_map_grouped(&kp.map_src[0], source, kp.Cout, kp.groups, rows,
                                                out_dt, kp.cw) != CONV_OK))
      return plan_memory_direct(pl);
  } else if (kp.epi_mode == 2) {
    for (int ph = 0; ph < kp.num_phases; ++ph)
      if (encode_out_map_phase(&kp.map_out[ph], output, kp, ph, n_images, out_dt, kp.cw) != CONV_OK ||
          (has_residual &&
           encode_out_map_phase(&kp.map_src[ph], source, kp, ph, n_images, out_dt, kp.cw) != CONV_OK))
        return plan_memory_direct(pl);
  }
  return CONV_OK;
}

// Direct-store epilogue: only the operand ring (and possibly the resident filter).
conv_status_t plan_memory_direct(Plan* pl) {
  ConvKernelParams& kp = pl->kp;
  const uint32_t a_bytes = kBM * kp.m_halves * kp.sw_bytes;
  const uint32_t b_bytes = static_cast<uint32_t>(kp.pair ? kp.bn / 2 : kp.bn) * kp.sw_bytes;
  const size_t bar_bytes = 1024 + gather_smem_bytes(kp);
  kp.epi_mode = 0;
  kp.cw = 16;
  kp.src_bufs = 0;
  kp.stg_bufs = 0;
  kp.src_chunk_bytes = 0;
  kp.valid_rows = kBM;
  const bool can_res = !kp.pair && !kp.streamk && kp.num_phases == 1 && kp.n_tiles == 1 &&
                       kp.groups <= 1;
  const size_t bres = can_res ? static_cast<size_t>(kp.taps_h[0]) * kp.taps_w[0] * kp.c_blocks * b_bytes : 0;
  // Few output channels with contiguous rows: staged 16-byte stores.
  kp.seg_store = (!kp.vec_ok && kp.num_phases == 1 && kp.out_step_h == 1 && kp.out_step_w == 1 &&
                  kp.groups <= 1 && kp.n_tiles == 1 && kp.bn == 16 && kp.Cout <= 16 && !kp.pair)
                     ? 1 : 0;
  kp.seg_slot_bytes = static_cast<uint32_t>((32 * 16 * 2 + 16 + 15) & ~15);
  const size_t seg_bytes = kp.seg_store ? align1k(static_cast<size_t>(4) * 2 * kp.seg_slot_bytes) : 0;
  bool res = false;
  int stages = 0;
  if (can_res) {
    const size_t used = 1024 + bar_bytes + align1k(bres) + seg_bytes;
    if (used + 4 * static_cast<size_t>(a_bytes) <= kSmemLimit) {
      res = true;
      stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - used) / a_bytes));
    }
  }
  if (!res) {
    const size_t used = 1024 + bar_bytes + seg_bytes;
    stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - used) / (a_bytes + b_bytes)));
    if (stages < 2) return CONV_ERR_NOT_SUPPORTED;
  }
  kp.b_resident = res ? 1 : 0;
  kp.stages = stages;
  uint32_t off = 0;
  kp.off_a = 0;
  off += align1k(static_cast<size_t>(stages) * a_bytes);
  kp.off_b = off;
  if (!res) off += align1k(static_cast<size_t>(stages) * b_bytes);
  kp.off_bres = off;
  if (res) off += align1k(bres);
  kp.off_seg = off;
  off += static_cast<uint32_t>(seg_bytes);
  kp.off_src = off;
  kp.off_stg = off;
  kp.off_bar = off;
  kp.off_gtab = off + 1024;
  kp.off_gstage = kp.off_gtab + align1k(static_cast<size_t>(kGatherProducers) * kBM * kp.m_halves * 16);
  off += bar_bytes;
  pl->smem_bytes = off + 1024;
  return CONV_OK;
}

// ------------------------------------------------------------------ launch
// Completes the kernel parameters of an implicit-GEMM plan: the filter and
// epilogue tensor maps, the shared-memory layout, the epilogue arguments and
// the grid.  No launch: the result may be cached and launched many times.
conv_status_t finish_plan(Plan* pl, int n_images, const void* packed, void* output,
                          int has_residual, const void* source, float beta,
                          conv_epilogue_t epilogue, void* workspace) {
  ConvKernelParams& kp = pl->kp;
  if (kp.groups < 1) {  // plans without channel groups
    kp.groups = 1;
    kp.c_group = kp.c_in;
    kp.f_group = kp.Cout;
    kp.tiles_per_group = kp.total_tiles;
  }
  // Filter slots: the stride phases, or the channel groups ([G][C_out/G][K]).
  conv_status_t st =
      kp.groups > 1
          ? encode_filter_map(&kp.map_b, packed, pl->kmax, kp.f_group, kp.groups, pl->in_dtype,
                              kp.bk, kp.bn, kp.sw_bytes)
          : encode_filter_map(&kp.map_b, packed, pl->kmax, kp.Cout, pl->phases_packed,
                              pl->in_dtype, kp.bk, kp.pair ? kp.bn / 2 : kp.bn, kp.sw_bytes);
  if (st != CONV_OK) return st;
  st = plan_memory(pl, n_images, output, has_residual ? source : nullptr, has_residual);
  if (st != CONV_OK) return st;
  kp.has_residual = has_residual ? 1 : 0;
  kp.src = has_residual ? source : nullptr;
  kp.beta = has_residual ? beta : 0.0f;
  kp.epilogue = static_cast<int>(epilogue);
  kp.out = output;
  kp.status = static_cast<unsigned int*>(workspace);
  const unsigned long long tmo = g_timeout_ns.load(std::memory_order_relaxed);
  kp.timeout_cycles = ns_to_cycles(tmo ? tmo : kDefaultTimeoutNs);
  kp.wait_hint_ns = tuning().wait_hint_ns;
  kp.fault_mode = g_fault_mode.load(std::memory_order_relaxed);
  // Two MMA issuers, one per 128-row half, where there are two halves and
  // warp 11 is free (TMA loaders, single CTAs).  CONV_MMA_SPLIT=0 disables.
  kp.mma_split = (kp.m_halves == 2 && !kp.gather && !kp.pair && tuning().mma_split != 0) ? 1 : 0;
  kp.div_ntiles = make_fast_div(static_cast<uint32_t>(std::max(kp.n_tiles, 1)));
  for (int ph = 0; ph < kMaxPhases; ++ph) {
    const uint32_t gh = static_cast<uint32_t>(std::max(kp.grid_h[ph], 1));
    const uint32_t gw = static_cast<uint32_t>(std::max(kp.grid_w[ph], 1));
    kp.div_ghw[ph] = make_fast_div(gh * gw);
    kp.div_gw[ph] = make_fast_div(gw);
  }
  kp.div_win_rb = make_fast_div(static_cast<uint32_t>(std::max(kp.win_row_blocks, 1)));
  kp.div_tpg = make_fast_div(static_cast<uint32_t>(std::max(kp.tiles_per_group, 1)));
  // Prefetching the next tile's input only pays when CTAs walk several tiles
  // that all start at the first C_out tile (one n-tile).
  kp.l2_prefetch = (kp.n_tiles == 1 && !kp.streamk && tuning().l2_prefetch != -1) ? 1 : 0;
  const int sms = device_sm_count();
  if (sms <= 0) return CONV_ERR_CUDA;
  // Pairs: clusters of two CTAs, one tile per cluster at a time.  Stream-K:
  // one CTA per SM, each with its share of the iterations.
  pl->grid = kp.pair ? 2 * std::min(kp.total_tiles, sms / 2)
                     : (kp.streamk ? sms : std::min(kp.total_tiles, sms));
  if (kp.streamk) {
    uint8_t* base = static_cast<uint8_t*>(workspace) + pl->sk_offset;
    kp.sk_flags = reinterpret_cast<unsigned int*>(base);
    kp.sk_partials = reinterpret_cast<float*>(base + sk_flag_bytes(pl->grid));
  }
  return CONV_OK;
}

conv_status_t launch_plan(const Plan& pl, cudaStream_t stream) {
  if (pl.kp.total_tiles == 0) return CONV_OK;
  cudaError_t e = launch_conv_igemm(pl.kind, pl.out_bf16, pl.kp, pl.grid, pl.smem_bytes, stream);
  return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

// ------------------------------------------------------------------ row-tap path
// Forward convs with few output channels (S * C_out <= 32): the filter taps
// along S and the output channels share the MMA's N dimension, each input row
// segment is loaded and multiplied once, and the R filter rows accumulate into
// R output rows in tensor memory (conv_rowtap.cu).  Gate: one channel group,
// stride 1, dilation 1, a filter of more than one tap, 128-byte channel
// blocks (C_in * elt a multiple of 128), R * g16 <= 256 columns and a band of
// at least one row.  CONV_ROWTAP=-1 disables it; CONV_ROWTAP_BAND sets the
// band height (output rows per tile, capped by the TMEM columns).
struct RowTapPlan {
  RowTapParams rp;
  int grid;
  size_t smem_bytes;
  int in_dtype;
};

bool plan_rowtap(const FwdShape& f, int groups, int num_sms, RowTapPlan* out) {
  if (tuning().rowtap == -1) return false;
  if (groups != 1 || f.stride_h != 1 || f.stride_w != 1 || f.dil_h != 1 || f.dil_w != 1)
    return false;
  if (f.r * f.s < 2) return false;
  const int elt = elt_bytes(f.in_dtype);
  if ((static_cast<long long>(f.c_in) * elt) % 128 != 0) return false;
  const int sf = f.s * f.c_out;
  if (sf > 32) return false;
  const int g16 = sf <= 16 ? 16 : 32;
  if (f.r * g16 > 256) return false;
  // Columns per accumulator buffer: g16 * (band + 2R - 2).  Two buffers
  // (<= 256 columns each) let a CTA's next tile start while its epilogue
  // drains; when every CTA has one tile, one buffer of up to 512 columns
  // allows taller bands.
  const int band_max2 = std::min(kRowTapMaxBand, 256 / g16 - 2 * f.r + 2);
  const int band_max1 = std::min(kRowTapMaxBand, 512 / g16 - 2 * f.r + 2);
  if (band_max1 < 1) return false;
  const int seg_w = 128 - (f.s - 1);
  const int n_seg = (f.wo + seg_w - 1) / seg_w;
  auto tiles_of = [&](int b) {
    return static_cast<long long>(f.n) * ((f.ho + b - 1) / b) * n_seg;
  };
  auto fits = [&](int b) { return b <= band_max2 || tiles_of(b) <= num_sms; };
  // Band height: the fewest input-row loads on the busiest SM (each tile
  // loads band + R - 1 rows); ties go to the taller band.
  int best = 0;
  long long best_cost = -1;
  for (int b = 1; b <= band_max1; ++b) {
    if (!fits(b)) continue;
    const long long waves = (tiles_of(b) + num_sms - 1) / num_sms;
    const long long cost = waves * (b + f.r - 1);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best = b;
    }
  }
  if (best == 0) return false;
  const int band_env = tuning().rowtap_band;  // tuning override: output rows per tile
  if (band_env > 0) {
    best = std::min(band_env, band_max1);
    while (best > 1 && !fits(best)) --best;
  }
  const int n_band = (f.ho + best - 1) / best;
  const long long tiles = static_cast<long long>(f.n) * n_band * n_seg;
  const bool one_buffer = best > band_max2;  // (then every CTA has one tile)
  if (tiles >= (1ll << 31)) return false;
  std::memset(out, 0, sizeof(*out));
  RowTapParams& rp = out->rp;
  rp.N = f.n; rp.H = f.h; rp.W = f.w; rp.Ho = f.ho; rp.Wo = f.wo;
  rp.F = f.c_out; rp.R = f.r; rp.S = f.s;
  rp.pad_h = f.pad_h; rp.pad_w = f.pad_w;
  rp.c_blocks = static_cast<int>((static_cast<long long>(f.c_in) * elt) / 128);
  rp.g16 = g16;
  rp.band = best;
  rp.seg_w = seg_w;
  rp.n_seg = n_seg;
  rp.n_band = n_band;
  rp.total_tiles = static_cast<int>(tiles);
  rp.idesc_all = make_idesc(f.in_dtype, f.r * g16);
  rp.idesc_one = make_idesc(f.in_dtype, g16);
  rp.idesc_rest = make_idesc(f.in_dtype, std::max(f.r - 1, 1) * g16);
  rp.cols_per_buf = static_cast<uint32_t>(g16 * (best + 2 * f.r - 2));
  rp.tmem_cols = next_pow2_cols(static_cast<int>((one_buffer ? 1 : 2) * rp.cols_per_buf));
  // Shared memory: the A ring at 0, the resident filter, the epilogue's
  // exchange buffers (two groups x two rows), the barriers.  An A stage holds
  // every channel block of one input row segment when four such stages fit
  // (one wait and one commit per input row instead of per block: the RGB
  // head's MMA warp spent ~560 cycles per 16 KB stage), else one block.
  const size_t blk_bytes = 128 * 128;
  const size_t b_bytes = static_cast<size_t>(rp.c_blocks) * f.r * g16 * 128;
  const size_t part_bytes = static_cast<size_t>(2 * 2) * g16 * 128 * sizeof(float);
  // Row-segment stages of the epilogue: output and source, per group.
  const int seg_stage = static_cast<int>((static_cast<size_t>(128) * f.c_out * 2 + 16 + 15) & ~size_t(15));
  const size_t seg_bytes = static_cast<size_t>(4) * seg_stage;
  const size_t fixed = 1024 + align1k(b_bytes) + align1k(part_bytes) + align1k(seg_bytes) + 1024;
  int blocks = rp.c_blocks;
  if (tuning().rowtap_blocks == 1 || fixed + 4 * blocks * blk_bytes > kSmemLimit) blocks = 1;
  const size_t stage_bytes = blocks * blk_bytes;
  rp.blocks_per_stage = blocks;
  if (fixed + 2 * stage_bytes > kSmemLimit) return false;
  rp.stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - fixed) / stage_bytes));
  rp.off_b = static_cast<uint32_t>(rp.stages * stage_bytes);
  rp.off_part = rp.off_b + align1k(b_bytes);
  rp.off_stage = rp.off_part + align1k(part_bytes);
  rp.stage_bytes = seg_stage;
  rp.off_bar = rp.off_stage + align1k(seg_bytes);
  out->smem_bytes = 1024 + rp.off_bar + 1024;
  out->grid = static_cast<int>(std::min<long long>(tiles, num_sms));
  return true;
}

// Encodes the row-tap kernel's maps and fills its epilogue arguments (no launch).
conv_status_t finish_rowtap(RowTapPlan* pl, const FwdShape& f, const void* input,
                            const void* packed, void* output, int has_residual,
                            const void* source, float beta, conv_epilogue_t epilogue,
                            void* workspace) {
  const DriverFns* fns = driver_fns();
  if (!fns) return CONV_ERR_CUDA;
  RowTapParams& rp = pl->rp;
  const cuuint64_t e = static_cast<cuuint64_t>(elt_bytes(f.in_dtype));
  const cuuint32_t bk = static_cast<cuuint32_t>(128 / e);
  {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(f.c_in), static_cast<cuuint64_t>(f.w),
                          static_cast<cuuint64_t>(f.h), static_cast<cuuint64_t>(f.n)};
    cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
    cuuint32_t box[4] = {bk, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fns->tiled(&rp.map_x, tmap_dtype(f.in_dtype), 4, const_cast<void*>(input), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CONV_ERR_CUDA;
  }
  {
    // The packed filter [F][(r*S + s)*C_in + c] seen as {C_in, S, R, F}.
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(f.c_in), static_cast<cuuint64_t>(f.s),
                          static_cast<cuuint64_t>(f.r), static_cast<cuuint64_t>(f.c_out)};
    cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
    cuuint32_t box[4] = {bk, static_cast<cuuint32_t>(f.s), 1, static_cast<cuuint32_t>(f.c_out)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fns->tiled(&rp.map_w, tmap_dtype(f.in_dtype), 4, const_cast<void*>(packed), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CONV_ERR_CUDA;
  }
  rp.has_residual = has_residual ? 1 : 0;
  rp.src = has_residual ? source : nullptr;
  rp.beta = has_residual ? beta : 0.0f;
  rp.epilogue = static_cast<int>(epilogue);
  rp.out = output;
  rp.status = static_cast<unsigned int*>(workspace);
  const unsigned long long tmo = g_timeout_ns.load(std::memory_order_relaxed);
  rp.timeout_cycles = ns_to_cycles(tmo ? tmo : kDefaultTimeoutNs);
  rp.fault_mode = g_fault_mode.load(std::memory_order_relaxed);
  pl->in_dtype = static_cast<int>(f.in_dtype);
  return CONV_OK;
}

conv_status_t launch_rowtap(const RowTapPlan& pl, cudaStream_t stream) {
  if (pl.rp.total_tiles == 0) return CONV_OK;
  cudaError_t err = launch_conv_rowtap(pl.in_dtype, pl.in_dtype != CONV_DTYPE_F16, pl.rp, pl.grid,
                                       pl.smem_bytes, stream);
  return err == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

bool epilogue_ok(conv_epilogue_t e) {
  return e == CONV_EPI_NONE || e == CONV_EPI_RELU || e == CONV_EPI_SILU;
}

conv_status_t check_common_ptrs(const void* input, const void* filter, void* output,
                                int has_residual, const void* source, void* workspace) {
  if (!input || !filter || !output || !workspace) return CONV_ERR_INVALID_VALUE;
  if (has_residual && !source) return CONV_ERR_INVALID_VALUE;
  if (!aligned16(input) || !aligned16(filter) || !aligned16(output) || !aligned16(workspace))
    return CONV_ERR_MISALIGNED;
  if (has_residual && !aligned16(source)) return CONV_ERR_MISALIGNED;
  return CONV_OK;
}

size_t round_up_256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

FwdShape make_fwd_shape(int n, int h, int w, int c_in, conv_dtype_t in_dtype, int r, int s,
                        int c_out, int ho, int wo, conv_dtype_t out_dtype, const int stride[2],
                        const int dilation[2], const int pad[2]) {
  FwdShape f{};
  f.n = n; f.h = h; f.w = w; f.c_in = c_in; f.r = r; f.s = s; f.c_out = c_out; f.ho = ho; f.wo = wo;
  f.stride_h = stride[0]; f.stride_w = stride[1];
  f.pad_h = pad[0]; f.pad_w = pad[1];
  f.dil_h = dilation[0]; f.dil_w = dilation[1];
  f.groups = 1;
  f.in_dtype = in_dtype; f.out_dtype = out_dtype;
  return f;
}

TrShape make_tr_shape(int n, int h, int w, int c_in, conv_dtype_t in_dtype, int r, int s,
                      int c_out, int ho, int wo, conv_dtype_t out_dtype, const int stride[2],
                      const int dilation[2], const int pad[2]) {
  TrShape t{};
  t.n = n; t.h = h; t.w = w; t.c_in = c_in; t.r = r; t.s = s; t.c_out = c_out; t.ho = ho; t.wo = wo;
  t.stride_h = stride[0]; t.stride_w = stride[1];
  t.pad_h = pad[0]; t.pad_w = pad[1];
  t.dil_h = dilation[0]; t.dil_w = dilation[1];
  t.in_dtype = in_dtype; t.out_dtype = out_dtype;
  return t;
}

// A call made ready to launch: which kernel runs it, its complete parameters
// (tensor maps encoded, shared memory laid out, grid chosen) and, for the
// entry points that take a raw filter, the packing launch that precedes it.
enum { kPathIgemm = 0, kPathRowTap = 1, kPathDirect = 2 };

struct PackStep {
  int kind;                 // 0 none, 1 forward filter, 2 transposed filter
  const void* filter;
  void* dst;
  int r, s, c_in, c_out, fcrs;
  conv_dtype_t dtype;
};

struct Prepared {
  int path;
  PackStep pack;
  TrPacking trp;    // transposed convs: the packed filter's layout (for the pack step)
  // kPathIgemm: the launches, in order (one, or for a transposed conv with
  // more than kMaxPhases phase slots, one per group of kMaxPhases slots; the
  // groups write disjoint output pixels).
  int n_plans;
  Plan pl[kMaxTrLaunches];
  RowTapPlan rt;    // kPathRowTap
  DirectParams dp;  // kPathDirect
  int direct_in_dtype;
  int sms;
};

conv_status_t run_pack(const Prepared& pr, cudaStream_t stream) {
  const PackStep& k = pr.pack;
  if (k.kind == 1)
    return launch_pack_fwd(k.filter, k.r, k.s, k.c_in, k.c_out, k.fcrs, k.dtype, k.dst, stream);
  if (k.kind == 2)
    return launch_pack_tr(pr.trp, k.filter, k.r, k.s, k.c_in, k.c_out, k.dtype, k.dst, stream);
  return CONV_OK;
}

// Stream-K flags hold the value of the launch that raised them: every launch
// takes a new value (never 0, the value of a fresh workspace), so flags left
// by an earlier launch -- finished or stopped by a timeout -- never match.
std::atomic<uint32_t> g_sk_epoch{0};

uint32_t next_sk_epoch() {
  uint32_t e;
  do {
    e = g_sk_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  } while (e == 0);
  return e;
}

conv_status_t launch_prepared(const Prepared& pr, cudaStream_t stream) {
  conv_status_t st = run_pack(pr, stream);
  if (st != CONV_OK) return st;
  if (pr.path == kPathRowTap) return launch_rowtap(pr.rt, stream);
  if (pr.path == kPathDirect) {
    cudaError_t e = launch_conv_direct(pr.direct_in_dtype, pr.direct_in_dtype != CONV_DTYPE_F16,
                                       pr.dp, pr.sms, stream);
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
  }
  for (int i = 0; i < pr.n_plans; ++i) {
    if (pr.pl[i].kp.streamk) {
      // The prepared plan is shared and immutable: the launch's flag value
      // goes into a copy.
      thread_local Plan sk_plan;
      sk_plan = pr.pl[i];
      sk_plan.kp.sk_epoch = next_sk_epoch();
      st = launch_plan(sk_plan, stream);
    } else {
      st = launch_plan(pr.pl[i], stream);
    }
    if (st != CONV_OK) return st;
  }
  return CONV_OK;
}

// Prepares conv2d_fwd / conv2d_fwd_packed.  `filter` is raw (packed into the
// workspace first) unless `prepacked`.
conv_status_t prepare_fwd(const void* input, const FwdShape& shape, const void* filter, int fcrs,
                          bool prepacked, void* output, int num_groups, int has_residual,
                          const void* source, float beta, conv_epilogue_t epilogue,
                          void* workspace, size_t workspace_bytes, Prepared* pr) {
  conv_status_t st = check_common_ptrs(input, filter, output, has_residual, source, workspace);
  if (st != CONV_OK) return st;
  if (!epilogue_ok(epilogue)) return CONV_ERR_INVALID_VALUE;
  st = check_fwd_shape(shape, num_groups);
  if (st != CONV_OK) return st;
  FwdShape f = shape;
  f.groups = num_groups;
  const int cg = f.c_in / num_groups;  // the filter's channel extent
  const size_t packed_bytes = conv2d_packed_filter_bytes(f.r, f.s, cg, f.c_out, f.in_dtype);
  const size_t need = CONV_STATUS_BYTES + (prepacked ? 0 : round_up_256(packed_bytes));
  if (workspace_bytes < need) return CONV_ERR_WORKSPACE_TOO_SMALL;
  const int sms = device_sm_count();
  if (sms <= 0) return CONV_ERR_CUDA;
  pr->sms = sms;
  const void* packed = filter;
  pr->pack.kind = 0;
  if (!prepacked) {
    void* dst = static_cast<uint8_t*>(workspace) + CONV_STATUS_BYTES;
    pr->pack = PackStep{1, filter, dst, f.r, f.s, cg, f.c_out, fcrs, f.in_dtype};
    packed = dst;
  }
  if (num_groups > 1 && !groups_on_tensor_cores(cg, elt_bytes(f.in_dtype))) {
    const int elt = elt_bytes(f.in_dtype);
    DirectParams& dp = pr->dp;
    dp = DirectParams{};
    dp.x = input;
    dp.w = packed;
    dp.src = has_residual ? source : nullptr;
    dp.y = output;
    dp.N = f.n; dp.H = f.h; dp.W = f.w; dp.C = f.c_in; dp.Ho = f.ho; dp.Wo = f.wo;
    dp.F = f.c_out; dp.R = f.r; dp.S = f.s;
    dp.c_group = cg;
    dp.f_group = f.c_out / num_groups;
    dp.stride_h = f.stride_h; dp.stride_w = f.stride_w;
    dp.pad_h = f.pad_h; dp.pad_w = f.pad_w;
    dp.dil_h = f.dil_h; dp.dil_w = f.dil_w;
    dp.w_runs = gather_mode(cg, elt) ? 1 : 0;
    dp.run_elems = static_cast<int>(gather_run_bytes(f.s, cg, elt) / elt);
    dp.kdim = static_cast<int>(fwd_packed_k(f.r, f.s, cg, elt));
    dp.has_residual = has_residual ? 1 : 0;
    dp.epilogue = static_cast<int>(epilogue);
    dp.beta = has_residual ? beta : 0.0f;
    dp.div_wo = make_fast_div(static_cast<uint32_t>(f.wo));
    dp.div_ho = make_fast_div(static_cast<uint32_t>(f.ho));
    dp.status = static_cast<unsigned int*>(workspace);
    const unsigned long long tmo = g_timeout_ns.load(std::memory_order_relaxed);
    dp.timeout_cycles = ns_to_cycles(tmo ? tmo : kDefaultTimeoutNs);
    dp.fault_mode = g_fault_mode.load(std::memory_order_relaxed);
    dp.dw_cols = dw_tile_cols(f.wo);
    if (direct_uses_dw_tiles(static_cast<int>(f.in_dtype), dp)) {
      // Depthwise 3x3 tiles: {C, W, H, N} boxes of kDwRows + 2 rows x dw_cols + 2
      // columns x 64 channels, zero outside the image.
      const DriverFns* fns = driver_fns();
      if (!fns) return CONV_ERR_CUDA;
      const cuuint64_t e = static_cast<cuuint64_t>(elt);
      cuuint64_t dims[4] = {static_cast<cuuint64_t>(f.c_in), static_cast<cuuint64_t>(f.w),
                            static_cast<cuuint64_t>(f.h), static_cast<cuuint64_t>(f.n)};
      cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
      cuuint32_t box[4] = {64, static_cast<cuuint32_t>(dp.dw_cols + 2), kDwRows + 2, 1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      if (fns->tiled(&dp.map_x, tmap_dtype(f.in_dtype), 4, const_cast<void*>(input), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return CONV_ERR_CUDA;
    }
    pr->path = kPathDirect;
    pr->direct_in_dtype = static_cast<int>(f.in_dtype);
    return CONV_OK;
  }
  if (plan_rowtap(f, num_groups, sms, &pr->rt)) {
    pr->path = kPathRowTap;
    return finish_rowtap(&pr->rt, f, input, packed, output, has_residual, source, beta, epilogue,
                         workspace);
  }
  Plan& pl = pr->pl[0];
  pr->n_plans = 1;
  const size_t sk_offset = need;
  st = plan_fwd(f, &pl, sms, has_residual,
                workspace_bytes > sk_offset ? workspace_bytes - sk_offset : 0);
  if (st != CONV_OK) return st;
  pl.sk_offset = sk_offset;
  st = encode_fwd_input(f, input, &pl);
  if (st != CONV_OK) return st;
  pr->path = kPathIgemm;
  return finish_plan(&pl, f.n, packed, output, has_residual, source, beta, epilogue, workspace);
}

conv_status_t prepare_tr(const void* input, const TrShape& t, const void* filter, bool prepacked,
                         void* output, int has_residual, const void* source, float beta,
                         conv_epilogue_t epilogue, void* workspace, size_t workspace_bytes,
                         Prepared* pr) {
  conv_status_t st = check_common_ptrs(input, filter, output, has_residual, source, workspace);
  if (st != CONV_OK) return st;
  if (!epilogue_ok(epilogue)) return CONV_ERR_INVALID_VALUE;
  st = check_tr_shape(t);
  if (st != CONV_OK) return st;
  int bk = 0;
  uint32_t row_bytes = 0;
  st = channel_block(t.c_in, elt_bytes(t.in_dtype), &bk, &row_bytes);
  if (st != CONV_OK) return st;
  const int st_hw[2] = {t.stride_h, t.stride_w};
  const int dil_hw[2] = {t.dil_h, t.dil_w};
  const int pad_hw[2] = {t.pad_h, t.pad_w};
  if (!tr_packing(t.r, t.s, t.c_in, st_hw, dil_hw, pad_hw, &pr->trp)) return CONV_ERR_NOT_SUPPORTED;
  const size_t packed_bytes =
      static_cast<size_t>(pr->trp.slots) * t.c_out * pr->trp.kmax * elt_bytes(t.in_dtype);
  const size_t need = CONV_STATUS_BYTES + (prepacked ? 0 : round_up_256(packed_bytes));
  if (workspace_bytes < need) return CONV_ERR_WORKSPACE_TOO_SMALL;
  const int sms = device_sm_count();
  if (sms <= 0) return CONV_ERR_CUDA;
  pr->sms = sms;
  const void* packed = filter;
  pr->pack.kind = 0;
  if (!prepacked) {
    void* dst = static_cast<uint8_t*>(workspace) + CONV_STATUS_BYTES;
    pr->pack = PackStep{2, filter, dst, t.r, t.s, t.c_in, t.c_out, 0, t.in_dtype};
    packed = dst;
  }
  pr->path = kPathIgemm;
  // Phase slots with output pixels, kMaxPhases per launch.
  int slots[kMaxTrSlots];
  const int nslots = tr_active_slots(t, slots);
  pr->n_plans = (nslots + kMaxPhases - 1) / kMaxPhases;
  const size_t sk_offset = need;
  for (int i = 0; i < pr->n_plans; ++i) {
    Plan& pl = pr->pl[i];
    st = plan_transposed(t, pr->trp, slots + i * kMaxPhases,
                         std::min(kMaxPhases, nslots - i * kMaxPhases), &pl, sms,
                         workspace_bytes > sk_offset ? workspace_bytes - sk_offset : 0);
    if (st != CONV_OK) return st;
    pl.sk_offset = sk_offset;
    st = encode_tr_inputs(t, input, &pl);
    if (st != CONV_OK) return st;
    st = finish_plan(&pl, t.n, packed, output, has_residual, source, beta, epilogue, workspace);
    if (st != CONV_OK) return st;
  }
  return CONV_OK;
}

// ------------------------------------------------------------------ prepared-call cache
// Planning and tensor-map encoding cost microseconds of host time per call;
// a call repeated with the same arguments (pointers included: a tensor map
// holds the address) reuses the prepared launch.  The key holds every
// argument plus the device, the tuning generation and the test hooks, so an
// entry is valid exactly when a fresh preparation would produce it.
struct CallKey {
  int entry;  // 0 conv2d_fwd, 1 conv2d_fwd_packed, 2 conv_transposed, 3 conv_transposed_packed
  int device;
  unsigned tuning_gen;
  int fault_mode;
  unsigned long long timeout_ns;
  const void* ptrs[5];  // input, filter, output, source, workspace
  size_t workspace_bytes;
  int dims[20];
  uint32_t beta_bits;
};

// Open addressing: a key's home slot is its hash modulo the table size and
// it may sit in any of the kProbe slots from there; a store into a full
// window replaces the slot after the one replaced last.
constexpr int kCacheEntries = 1024;
constexpr int kProbe = 8;
struct CacheSlot {
  bool valid;
  CallKey key;
  std::shared_ptr<const Prepared> prep;  // immutable once stored
};

std::mutex g_cache_mu;
CacheSlot* g_cache = nullptr;  // kCacheEntries slots, allocated on first use
int g_cache_victim = 0;
std::atomic<unsigned long long> g_cache_hits{0}, g_cache_misses{0};

uint64_t key_hash(const CallKey& key) {
  // FNV-1a over the key's bytes (padding included: keys are zero-filled).
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&key);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof(key); ++i) {
    h ^= b[i];
    h *= 1099511628211ull;
  }
  return h;
}

CallKey make_key(int entry, const void* input, const void* filter, const void* output,
                 const void* source, const void* workspace, size_t workspace_bytes, int n, int h,
                 int w, int c_in, conv_dtype_t in_dtype, int r, int s, int c_out, int fcrs, int ho,
                 int wo, conv_dtype_t out_dtype, const int stride[2], const int dilation[2],
                 const int pad[2], int num_groups, int has_residual, float beta,
                 conv_epilogue_t epilogue) {
  CallKey k;
  std::memset(&k, 0, sizeof(k));  // padding bytes take part in the comparison
  k.entry = entry;
  if (cudaGetDevice(&k.device) != cudaSuccess) k.device = -1;
  tuning();  // loads the overrides on first use, so the generation below is final
  k.tuning_gen = g_tuning_gen.load(std::memory_order_acquire);
  k.fault_mode = g_fault_mode.load(std::memory_order_relaxed);
  k.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  k.ptrs[0] = input;
  k.ptrs[1] = filter;
  k.ptrs[2] = output;
  k.ptrs[3] = has_residual ? source : nullptr;
  k.ptrs[4] = workspace;
  k.workspace_bytes = workspace_bytes;
  const int d[20] = {n, h, w, c_in, static_cast<int>(in_dtype), r, s, c_out, fcrs, ho, wo,
                     static_cast<int>(out_dtype), stride[0], stride[1], dilation[0], dilation[1],
                     pad[0], pad[1], num_groups, has_residual ? 1 : 0};
  std::memcpy(k.dims, d, sizeof(d));
  const float b = has_residual ? beta : 0.0f;
  std::memcpy(&k.beta_bits, &b, sizeof(b));
  k.dims[19] |= static_cast<int>(epilogue) << 8;
  return k;
}

std::shared_ptr<const Prepared> cache_lookup(const CallKey& key) {
  const size_t home = key_hash(key) % kCacheEntries;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  if (g_cache) {
    for (int i = 0; i < kProbe; ++i) {
      const CacheSlot& slot = g_cache[(home + i) % kCacheEntries];
      if (slot.valid && std::memcmp(&slot.key, &key, sizeof(key)) == 0) {
        g_cache_hits.fetch_add(1, std::memory_order_relaxed);
        return slot.prep;
      }
    }
  }
  g_cache_misses.fetch_add(1, std::memory_order_relaxed);
  return nullptr;
}

void cache_store(const CallKey& key, const std::shared_ptr<const Prepared>& prep) {
  const size_t home = key_hash(key) % kCacheEntries;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  if (!g_cache) {
    g_cache = new (std::nothrow) CacheSlot[kCacheEntries];
    if (!g_cache) return;  // no cache: every call prepares afresh
    for (int i = 0; i < kCacheEntries; ++i) g_cache[i].valid = false;
  }
  int pick = -1;
  for (int i = 0; i < kProbe && pick < 0; ++i)
    if (!g_cache[(home + i) % kCacheEntries].valid) pick = i;
  if (pick < 0) {
    pick = g_cache_victim;
    g_cache_victim = (g_cache_victim + 1) % kProbe;
  }
  CacheSlot& slot = g_cache[(home + pick) % kCacheEntries];
  slot.key = key;
  slot.prep = prep;
  slot.valid = true;
}

// Looks the call up, prepares it on a miss (caching only successful
// preparations), and launches it.
template <typename PrepareFn>
conv_status_t cached_call(const CallKey& key, PrepareFn prepare, cudaStream_t stream) {
  std::shared_ptr<const Prepared> pr = cache_lookup(key);
  if (!pr) {
    // Large (several plans): on the heap, zero-initialised.
    std::shared_ptr<Prepared> fresh(new (std::nothrow) Prepared());
    if (!fresh) return CONV_ERR_INVALID_VALUE;
    conv_status_t st = prepare(fresh.get());
    if (st != CONV_OK) return st;
    if (key.device >= 0) cache_store(key, fresh);
    pr = fresh;
  }
  return launch_prepared(*pr, stream);
}

}  // namespace

namespace {

// ------------------------------------------------------------------ no-allocation variant
// Scratch for conv2d_fwd_noalloc: the status word and the packed filter live
// in this file-scope device array instead of a caller-provided workspace.
// Every GPU that loads the library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current device's context (host
// code must not use the symbol itself as a pointer).  Looked up on every call:
// the lookup is host-only and cheap, and an address cached across calls could
// outlive the context it belongs to (after cudaDeviceReset, say).
void* noalloc_scratch_ptr(conv_status_t* st) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    *st = CONV_ERR_CUDA;
    return nullptr;
  }
  *st = CONV_OK;
  return p;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* conv_status_string(conv_status_t status) {
  switch (status) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_INVALID_VALUE: return "CONV_ERR_INVALID_VALUE";
    case CONV_ERR_NOT_SUPPORTED: return "CONV_ERR_NOT_SUPPORTED";
    case CONV_ERR_MISALIGNED: return "CONV_ERR_MISALIGNED";
    case CONV_ERR_WORKSPACE_TOO_SMALL: return "CONV_ERR_WORKSPACE_TOO_SMALL";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA";
    case CONV_ERR_DEVICE_TIMEOUT: return "CONV_ERR_DEVICE_TIMEOUT";
  }
  return "CONV_ERR_UNKNOWN";
}

size_t conv2d_packed_filter_bytes(int r, int s, int c_in, int c_out, conv_dtype_t dtype) {
  if (r <= 0 || s <= 0 || c_in <= 0 || c_out <= 0 || !known_dtype(dtype)) return 0;
  const int elt = elt_bytes(dtype);
  return static_cast<size_t>(fwd_packed_k(r, s, c_in, elt)) * c_out * elt;
}

size_t conv2d_workspace_size(int r, int s, int c_in, int c_out, conv_dtype_t dtype) {
  return CONV_STATUS_BYTES + round_up_256(conv2d_packed_filter_bytes(r, s, c_in, c_out, dtype));
}

size_t conv_streamk_workspace_size(void) {
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // The largest tile: 128 x 256 or 256 x 128 fp32 accumulators.
  return sk_flag_bytes(sms) + static_cast<size_t>(sms) * (size_t(kBM) * 256 * sizeof(float));
}

conv_status_t conv2d_pack_filter(const void* filter, int r, int s, int c_in, int c_out,
                                 int filter_is_fcrs, conv_dtype_t dtype, void* packed,
                                 size_t packed_bytes, void* stream) {
  if (!filter || !packed) return CONV_ERR_INVALID_VALUE;
  if (r <= 0 || s <= 0 || c_in <= 0 || c_out <= 0) return CONV_ERR_INVALID_VALUE;
  if (!known_dtype(dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (!aligned16(filter) || !aligned16(packed)) return CONV_ERR_MISALIGNED;
  if (packed_bytes < conv2d_packed_filter_bytes(r, s, c_in, c_out, dtype))
    return CONV_ERR_WORKSPACE_TOO_SMALL;
  return launch_pack_fwd(filter, r, s, c_in, c_out, filter_is_fcrs ? 1 : 0, dtype, packed,
                         static_cast<cudaStream_t>(stream));
}

conv_status_t conv2d_fwd(const void* input, int n, int h, int w, int c_in, conv_dtype_t in_dtype,
                         const void* filter, int r, int s, int c_out, int filter_is_fcrs,
                         void* output, int ho, int wo, conv_dtype_t out_dtype,
                         const int stride[2], const int dilation[2],
                         const int symmetric_padding[2], int num_groups, int has_residual,
                         const void* source, float beta, conv_epilogue_t epilogue,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!stride || !dilation || !symmetric_padding) return CONV_ERR_INVALID_VALUE;
  const FwdShape f = make_fwd_shape(n, h, w, c_in, in_dtype, r, s, c_out, ho, wo, out_dtype,
                                    stride, dilation, symmetric_padding);
  const int fcrs = filter_is_fcrs ? 1 : 0;
  const CallKey key = make_key(0, input, filter, output, source, workspace, workspace_bytes, n, h,
                               w, c_in, in_dtype, r, s, c_out, fcrs, ho, wo, out_dtype, stride,
                               dilation, symmetric_padding, num_groups, has_residual, beta,
                               epilogue);
  return cached_call(key, [&](Prepared* pr) {
    return prepare_fwd(input, f, filter, fcrs, false, output, num_groups, has_residual, source,
                       beta, epilogue, workspace, workspace_bytes, pr);
  }, static_cast<cudaStream_t>(stream));
}

conv_status_t conv2d_fwd_packed(const void* input, int n, int h, int w, int c_in,
                                conv_dtype_t in_dtype, const void* packed_filter, int r, int s,
                                int c_out, void* output, int ho, int wo, conv_dtype_t out_dtype,
                                const int stride[2], const int dilation[2],
                                const int symmetric_padding[2], int num_groups, int has_residual,
                                const void* source, float beta, conv_epilogue_t epilogue,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!stride || !dilation || !symmetric_padding) return CONV_ERR_INVALID_VALUE;
  const FwdShape f = make_fwd_shape(n, h, w, c_in, in_dtype, r, s, c_out, ho, wo, out_dtype,
                                    stride, dilation, symmetric_padding);
  const CallKey key = make_key(1, input, packed_filter, output, source, workspace, workspace_bytes,
                               n, h, w, c_in, in_dtype, r, s, c_out, 0, ho, wo, out_dtype, stride,
                               dilation, symmetric_padding, num_groups, has_residual, beta,
                               epilogue);
  return cached_call(key, [&](Prepared* pr) {
    return prepare_fwd(input, f, packed_filter, 0, true, output, num_groups, has_residual, source,
                       beta, epilogue, workspace, workspace_bytes, pr);
  }, static_cast<cudaStream_t>(stream));
}

size_t conv_transposed_packed_filter_bytes_dilated(int r, int s, int c_in, int c_out,
                                                   const int stride[2], const int dilation[2],
                                                   const int padding[2], conv_dtype_t dtype) {
  if (!stride || !dilation || !padding || r <= 0 || s <= 0 || c_in <= 0 || c_out <= 0 ||
      !known_dtype(dtype))
    return 0;
  TrPacking pk;
  if (!tr_packing(r, s, c_in, stride, dilation, padding, &pk)) return 0;
  return static_cast<size_t>(pk.slots) * c_out * pk.kmax * elt_bytes(dtype);
}

size_t conv_transposed_packed_filter_bytes(int r, int s, int c_in, int c_out, const int stride[2],
                                           const int padding[2], conv_dtype_t dtype) {
  const int dil[2] = {1, 1};
  return conv_transposed_packed_filter_bytes_dilated(r, s, c_in, c_out, stride, dil, padding, dtype);
}

size_t conv_transposed_workspace_size_dilated(int r, int s, int c_in, int c_out,
                                              const int stride[2], const int dilation[2],
                                              const int padding[2], conv_dtype_t dtype) {
  return CONV_STATUS_BYTES + round_up_256(conv_transposed_packed_filter_bytes_dilated(
                                 r, s, c_in, c_out, stride, dilation, padding, dtype));
}

size_t conv_transposed_workspace_size(int r, int s, int c_in, int c_out, const int stride[2],
                                      const int padding[2], conv_dtype_t dtype) {
  const int dil[2] = {1, 1};
  return conv_transposed_workspace_size_dilated(r, s, c_in, c_out, stride, dil, padding, dtype);
}

conv_status_t conv_transposed_pack_filter_dilated(const void* filter_rsfc, int r, int s, int c_in,
                                                  int c_out, const int stride[2],
                                                  const int dilation[2], const int padding[2],
                                                  conv_dtype_t dtype, void* packed,
                                                  size_t packed_bytes, void* stream) {
  if (!filter_rsfc || !packed || !stride || !dilation || !padding) return CONV_ERR_INVALID_VALUE;
  if (r <= 0 || s <= 0 || c_in <= 0 || c_out <= 0) return CONV_ERR_INVALID_VALUE;
  if (!known_dtype(dtype)) return CONV_ERR_NOT_SUPPORTED;
  if (stride[0] < 1 || stride[1] < 1 || stride[0] * stride[1] > kMaxTrSlots)
    return CONV_ERR_NOT_SUPPORTED;
  if (dilation[0] < 1 || dilation[1] < 1 || dilation[0] > kMaxFilterExtent ||
      dilation[1] > kMaxFilterExtent)
    return CONV_ERR_NOT_SUPPORTED;
  if (padding[0] < 0 || padding[1] < 0 || padding[0] > dilation[0] * (r - 1) ||
      padding[1] > dilation[1] * (s - 1))
    return CONV_ERR_NOT_SUPPORTED;
  if (!aligned16(filter_rsfc) || !aligned16(packed)) return CONV_ERR_MISALIGNED;
  TrPacking pk;
  if (!tr_packing(r, s, c_in, stride, dilation, padding, &pk)) return CONV_ERR_NOT_SUPPORTED;
  if (packed_bytes < static_cast<size_t>(pk.slots) * c_out * pk.kmax * elt_bytes(dtype))
    return CONV_ERR_WORKSPACE_TOO_SMALL;
  return launch_pack_tr(pk, filter_rsfc, r, s, c_in, c_out, dtype, packed,
                        static_cast<cudaStream_t>(stream));
}

conv_status_t conv_transposed_pack_filter(const void* filter_rsfc, int r, int s, int c_in,
                                          int c_out, const int stride[2], const int padding[2],
                                          conv_dtype_t dtype, void* packed, size_t packed_bytes,
                                          void* stream) {
  const int dil[2] = {1, 1};
  return conv_transposed_pack_filter_dilated(filter_rsfc, r, s, c_in, c_out, stride, dil, padding,
                                             dtype, packed, packed_bytes, stream);
}

conv_status_t conv_transposed(const void* input, int n, int h, int w, int c_in,
                              conv_dtype_t in_dtype, const void* filter_rsfc, int r, int s,
                              int c_out, void* output, int ho, int wo, conv_dtype_t out_dtype,
                              const int stride[2], const int dilation[2], const int padding[2],
                              int has_residual, const void* source, float beta,
                              conv_epilogue_t epilogue, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!stride || !dilation || !padding) return CONV_ERR_INVALID_VALUE;
  const TrShape t = make_tr_shape(n, h, w, c_in, in_dtype, r, s, c_out, ho, wo, out_dtype, stride,
                                  dilation, padding);
  const CallKey key = make_key(2, input, filter_rsfc, output, source, workspace, workspace_bytes,
                               n, h, w, c_in, in_dtype, r, s, c_out, 0, ho, wo, out_dtype, stride,
                               dilation, padding, 1, has_residual, beta, epilogue);
  return cached_call(key, [&](Prepared* pr) {
    return prepare_tr(input, t, filter_rsfc, false, output, has_residual, source, beta, epilogue,
                      workspace, workspace_bytes, pr);
  }, static_cast<cudaStream_t>(stream));
}

conv_status_t conv_transposed_packed(const void* input, int n, int h, int w, int c_in,
                                     conv_dtype_t in_dtype, const void* packed_filter, int r,
                                     int s, int c_out, void* output, int ho, int wo,
                                     conv_dtype_t out_dtype, const int stride[2],
                                     const int dilation[2], const int padding[2], int has_residual,
                                     const void* source, float beta, conv_epilogue_t epilogue,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!stride || !dilation || !padding) return CONV_ERR_INVALID_VALUE;
  const TrShape t = make_tr_shape(n, h, w, c_in, in_dtype, r, s, c_out, ho, wo, out_dtype, stride,
                                  dilation, padding);
  const CallKey key = make_key(3, input, packed_filter, output, source, workspace, workspace_bytes,
                               n, h, w, c_in, in_dtype, r, s, c_out, 0, ho, wo, out_dtype, stride,
                               dilation, padding, 1, has_residual, beta, epilogue);
  return cached_call(key, [&](Prepared* pr) {
    return prepare_tr(input, t, packed_filter, true, output, has_residual, source, beta, epilogue,
                      workspace, workspace_bytes, pr);
  }, static_cast<cudaStream_t>(stream));
}

conv_status_t conv_check_device_status(void* workspace, void* stream, unsigned int* detail) {
  if (detail) *detail = 0;
  if (!workspace) return CONV_ERR_INVALID_VALUE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return CONV_ERR_CUDA;
  unsigned int bits = 0;
  if (cudaMemcpy(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CONV_ERR_CUDA;
  if (detail) *detail = bits;
  if (bits == 0) return CONV_OK;
  if (cudaMemset(workspace, 0, sizeof(bits)) != cudaSuccess) return CONV_ERR_CUDA;
  return CONV_ERR_DEVICE_TIMEOUT;
}

// See include/conv_gb300.h.  Validates the size against the scratch first
// (no CUDA call on rejection), resolves the scratch address of the current
// device, clears the status word, then runs the ordinary conv2d_fwd path with
// the scratch standing in for the workspace.
conv_status_t conv2d_fwd_noalloc(const void* input, int n, int h, int w, int c_in,
                                 conv_dtype_t in_dtype, const void* filter, int r, int s, int c_out,
                                 int filter_is_fcrs, void* output, int ho, int wo,
                                 conv_dtype_t out_dtype, const int stride[2], const int dilation[2],
                                 const int symmetric_padding[2], int num_groups, int has_residual,
                                 const void* source, float beta, conv_epilogue_t epilogue,
                                 void* stream) {
  if (r <= 0 || s <= 0 || c_in <= 0 || c_out <= 0 || !known_dtype(in_dtype))
    return CONV_ERR_INVALID_VALUE;
  if (num_groups < 1 || c_in % num_groups != 0) return CONV_ERR_INVALID_VALUE;
  // The packed filter spans C_in / num_groups channels, as in conv2d_fwd.
  const size_t need = conv2d_workspace_size(r, s, c_in / num_groups, c_out, in_dtype);
  if (need > kNoAllocScratchBytes) return CONV_ERR_WORKSPACE_TOO_SMALL;
  conv_status_t st = CONV_OK;
  void* scratch = noalloc_scratch_ptr(&st);
  if (st != CONV_OK) return st;
  if (cudaMemsetAsync(scratch, 0, CONV_STATUS_BYTES, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return CONV_ERR_CUDA;
  // The scratch stands in for a workspace of exactly conv2d_fwd's minimum
  // size, so the plan (and every result bit) is that of conv2d_fwd with such
  // a workspace.
  return conv2d_fwd(input, n, h, w, c_in, in_dtype, filter, r, s, c_out, filter_is_fcrs, output,
                    ho, wo, out_dtype, stride, dilation, symmetric_padding, num_groups,
                    has_residual, source, beta, epilogue, scratch, need, stream);
}

// ------------------------------------------------------------------- testing hooks
void conv_testing_set_wait_fault(int mode, unsigned long long timeout_ns) {
  g_fault_mode.store(mode, std::memory_order_relaxed);
  g_timeout_ns.store(timeout_ns, std::memory_order_relaxed);
}

void conv_testing_reload_tuning(void) {
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  g_tuning_value = read_tuning();
  const unsigned gen = g_tuning_gen.load(std::memory_order_relaxed);
  g_tuning_gen.store(gen + 1 == 0 ? 1 : gen + 1, std::memory_order_release);
}

void conv_testing_cache_stats(unsigned long long* hits, unsigned long long* misses) {
  if (hits) *hits = g_cache_hits.load(std::memory_order_relaxed);
  if (misses) *misses = g_cache_misses.load(std::memory_order_relaxed);
}

conv_status_t conv_testing_fwd_plan(int n, int h, int w, int c_in, conv_dtype_t dtype, int r,
                                    int s, int c_out, const int stride[2],
                                    const int symmetric_padding[2], int has_residual, int num_sms,
                                    size_t workspace_bytes, int out[14]) {
  if (!stride || !symmetric_padding || !out) return CONV_ERR_INVALID_VALUE;
  const int dil[2] = {1, 1};
  const conv_dtype_t out_dt = dtype == CONV_DTYPE_F8E4M3 ? CONV_DTYPE_BF16 : dtype;
  if (stride[0] <= 0 || stride[1] <= 0) return CONV_ERR_INVALID_VALUE;
  const int ho = (h + 2 * symmetric_padding[0] - (r - 1) - 1) / stride[0] + 1;
  const int wo = (w + 2 * symmetric_padding[1] - (s - 1) - 1) / stride[1] + 1;
  const FwdShape f = make_fwd_shape(n, h, w, c_in, dtype, r, s, c_out, ho, wo, out_dt, stride, dil,
                                    symmetric_padding);
  conv_status_t st = check_fwd_shape(f, 1);
  if (st != CONV_OK) return st;
  RowTapPlan rt;
  if (plan_rowtap(f, 1, num_sms, &rt)) {
    const RowTapParams& rp = rt.rp;
    out[0] = rp.R * rp.g16;
    out[1] = 128 / elt_bytes(dtype);
    out[2] = rp.stages;
    out[3] = static_cast<int>(rt.smem_bytes);
    out[4] = rp.total_tiles;
    out[5] = rt.grid;
    out[6] = static_cast<int>(rp.tmem_cols);
    out[7] = 0;
    out[8] = 1;
    out[9] = rp.blocks_per_stage;
    out[10] = rp.band;
    out[11] = 3;
    out[12] = 0;
    out[13] = 0;
    return CONV_OK;
  }
  Plan pl;
  st = plan_fwd(f, &pl, num_sms, has_residual,
                workspace_bytes > CONV_STATUS_BYTES ? workspace_bytes - CONV_STATUS_BYTES : 0);
  if (st != CONV_OK) return st;
  st = layout_memory(&pl, has_residual);
  if (st != CONV_OK) return st;
  out[0] = pl.kp.bn;
  out[1] = pl.kp.bk;
  out[2] = pl.kp.stages;
  out[3] = static_cast<int>(pl.smem_bytes);
  out[4] = pl.kp.total_tiles;
  out[5] = pl.kp.pair ? 2 * std::min(pl.kp.total_tiles, num_sms / 2)
                     : (pl.kp.streamk ? num_sms : std::min(pl.kp.total_tiles, num_sms));
  out[6] = static_cast<int>(pl.kp.tmem_cols);
  out[7] = pl.kp.epi_mode;
  out[8] = pl.kp.b_resident;
  out[9] = pl.kp.src_bufs;
  out[10] = pl.kp.stg_bufs;
  out[11] = pl.kp.gather ? 2 : (pl.kp.window ? 1 : 0);
  out[12] = pl.kp.pair;
  out[13] = pl.kp.streamk;
  return CONV_OK;
}

conv_status_t conv_testing_im2col_tile(const void* input, int n, int h, int w, int c_in,
                                       conv_dtype_t dtype, int r, int s, const int stride[2],
                                       const int symmetric_padding[2], int m0, int tap_r,
                                       int tap_s, int c0, void* out_tile, int* bk_out,
                                       void* status_workspace, void* stream) {
  if (!input || !out_tile || !status_workspace || !stride || !symmetric_padding)
    return CONV_ERR_INVALID_VALUE;
  if (!aligned16(input) || !aligned16(out_tile)) return CONV_ERR_MISALIGNED;
  const int dil[2] = {1, 1};
  const conv_dtype_t out_dt = dtype == CONV_DTYPE_F8E4M3 ? CONV_DTYPE_BF16 : dtype;
  if (stride[0] <= 0 || stride[1] <= 0) return CONV_ERR_INVALID_VALUE;
  const int ho = (h + 2 * symmetric_padding[0] - (r - 1) - 1) / stride[0] + 1;
  const int wo = (w + 2 * symmetric_padding[1] - (s - 1) - 1) / stride[1] + 1;
  const FwdShape f = make_fwd_shape(n, h, w, c_in, dtype, r, s, 16, ho, wo, out_dt, stride, dil,
                                    symmetric_padding);
  conv_status_t st = check_fwd_shape(f, 1);
  if (st != CONV_OK) return st;
  Plan pl;
  st = plan_fwd(f, &pl, 1, 0);
  if (st != CONV_OK) return st;
  if (pl.kp.gather) return CONV_ERR_NOT_SUPPORTED;  // no im2col map: plain loads build A
  pl.kp.m_halves = 1;  // the probe copies out one 128-row column of an im2col load
  pl.kp.window = 0;
  if (m0 < 0 || m0 >= pl.kp.rows[0] || tap_r < 0 || tap_r >= r || tap_s < 0 || tap_s >= s ||
      c0 < 0 || c0 >= c_in || c0 % pl.kp.bk != 0)
    return CONV_ERR_INVALID_VALUE;
  st = encode_fwd_input(f, input, &pl);
  if (st != CONV_OK) return st;
  const int hw = ho * wo;
  const int n_img = m0 / hw;
  const int rem = m0 - n_img * hw;
  const int j = rem / wo;
  const int i = rem - j * wo;
  const int h0 = -f.pad_h + j * f.stride_h;
  const int w0 = -f.pad_w + i * f.stride_w;
  if (bk_out) *bk_out = pl.kp.bk;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const unsigned long long tmo = g_timeout_ns.load(std::memory_order_relaxed);
  cudaError_t e = launch_im2col_probe(pl.kp.map_a[0], c0, w0, h0, n_img, tap_s, tap_r,
                                      pl.kp.sw_bytes, out_tile,
                                      static_cast<unsigned int*>(status_workspace),
                                      ns_to_cycles(tmo ? tmo : kDefaultTimeoutNs), cs);
  if (e != cudaSuccess) return CONV_ERR_CUDA;
  return cudaStreamSynchronize(cs) == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // extern "C"
