// Launch parameters shared by the host dispatcher and the implicit-GEMM
// kernel.  Passed by value as a __grid_constant__ kernel argument, so the
// tensor maps live in parameter space where TMA can read them.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace convgb300 {

constexpr int kBM = 128;             // rows (output pixels) per MMA = TMEM lanes
// Warps: 0 producer, 1 MMA, 2-9 epilogue, 10 producer, 11 producer (the gather
// loader: it builds A with three warps) or, with the TMA loaders and two
// 128-row halves per tile, the second MMA issuer.
constexpr int kThreads = 384;
constexpr int kProducer2Warp = 10;
constexpr int kProducer3Warp = 11;
constexpr int kGatherProducers = 3;
constexpr int kEpilogueWarps = 8;    // two warpgroups; each covers the 128 TMEM lanes once
constexpr int kEpilogueGroups = 2;
constexpr int kMaxPhases = 4;        // stride-phase GEMMs of a stride-2 transposed conv
constexpr int kMaxStages = 12;

constexpr int kKindF16 = 0;          // tcgen05.mma kind::f16 (bf16 or fp16 operands)
constexpr int kKindF8 = 1;           // tcgen05.mma kind::f8f6f4 (fp8 e4m3 operands)

constexpr int kEpiNone = 0;
constexpr int kEpiRelu = 1;
constexpr int kEpiSilu = 2;

// Device status bits (OR-ed into the workspace status word).
constexpr unsigned int kStatusProducerTimeout = 1u;
constexpr unsigned int kStatusMmaTimeout = 2u;
constexpr unsigned int kStatusEpilogueTimeout = 4u;
constexpr unsigned int kStatusStreamKTimeout = 8u;  // a stream-K partial never arrived

// Division by a fixed divisor d >= 1 as a multiply and shift, exact for
// 0 <= x < 2^31: q = (umulhi(x, mul) + x) >> shift with shift = ceil(log2 d)
// and mul = floor(2^32 * (2^shift - d) / d) + 1 (taken mod 2^32).
struct FastDiv {
  uint32_t d, mul, shift;
};

struct ConvKernelParams {  // aligned like CUtensorMap (64 B or more)
  CUtensorMap map_a[kMaxPhases];  // im2col maps over the NHWC input, one per phase
  CUtensorMap map_b;              // tiled map over the packed filter [phase][C_out][K]
  CUtensorMap map_out[kMaxPhases];  // TMA-store maps over the output (epilogue modes 1, 2)
  CUtensorMap map_src[kMaxPhases];  // TMA-load maps over the residual source (same boxes)

  int num_phases;
  int total_tiles;
  int pair;             // clusters of two CTAs share 256-row tiles (cta_group::2 MMAs)
  int mma_split;        // two MMA-issuing warps, one per 128-row half (m_halves = 2)
  int m_halves;         // 128-row halves per tile (1 or 2): tile_m = 128 * m_halves
  int n_tiles;          // tiles along C_out
  int bn;               // tile width along C_out (multiple of 16, <= 256)
  int bk;               // input channels per k-block
  int c_blocks;         // ceil(C_in / bk): channel blocks per filter tap
  int c_tail;           // C_in - c_blocks * bk (<= 0): k adjustment after a tap's last block
  int c_in;
  int stages;           // depth of the shared-memory ring
  uint32_t sw_bytes;    // bytes per operand row in a k-block (32, 64 or 128) = swizzle span
  uint32_t idesc;       // tcgen05 instruction descriptor
  uint32_t tmem_cols;   // allocated TMEM columns (two accumulators)
  uint32_t acc_stride;  // TMEM columns per accumulator buffer = m_halves * bn

  // Per phase: the output-pixel grid the GEMM rows walk, and where it reads.
  int tile_start[kMaxPhases + 1];  // first tile index of each phase (prefix sums)
  int rows[kMaxPhases];            // GEMM rows = N * grid_h * grid_w
  int grid_h[kMaxPhases];
  int grid_w[kMaxPhases];
  int taps_h[kMaxPhases];          // filter taps along H contributing to this phase
  int taps_w[kMaxPhases];
  int base_h[kMaxPhases];          // input row of grid row 0 at tap 0
  int base_w[kMaxPhases];
  int out_off_h[kMaxPhases];       // output row = out_step_h * grid row + out_off_h
  int out_off_w[kMaxPhases];
  int step_h, step_w;              // input rows/cols advanced per grid row/col
  int out_step_h, out_step_w;
  int dil_h, dil_w;                // input offset per filter tap
  int b_index[kMaxPhases];         // phase slot of the packed filter read by each phase
  // Channel groups (forward convs): output group g reads input channels
  // [g*c_group, (g+1)*c_group) through filter slot g and writes channels
  // [g*f_group, (g+1)*f_group).  Tiles are group-major:
  // t = g * tiles_per_group + (the tile within the group).
  int groups;
  int c_group, f_group;
  int tiles_per_group;
  // Division by the fixed divisors above, as multiply and shift (a runtime
  // integer division costs hundreds of cycles of latency).
  FastDiv div_ntiles;              // n_tiles
  FastDiv div_ghw[kMaxPhases];     // grid_h * grid_w
  FastDiv div_gw[kMaxPhases];      // grid_w
  FastDiv div_win_rb;              // win_row_blocks
  FastDiv div_tpg;                 // tiles_per_group

  // Shared-memory carve-up (byte offsets from the 1024-B aligned base).
  uint32_t off_a, off_b, off_bres, off_src, off_stg, off_bar;
  uint32_t off_gtab;               // gather loader: per-producer-warp row tables
  uint32_t off_gstage;             // gather loader: two input-row staging buffers
  int b_resident;                  // whole packed filter kept in shared memory (one phase, one n-tile)
  int l2_prefetch;                 // prefetch the next tile's A boxes into L2

  // Row-window A loader (stride-1 forward convs): a tile is win_rows output
  // rows per 128-row half; its input rows (with halo) arrive as one tiled box
  // [win_box_rows][win_pitch][bk] per channel block, and filter tap (r, s)
  // reads it from row r*win_pitch + s on.  win_pitch = Wo + S - 1 <= 128.
  int window;
  int win_pitch;
  int win_rows;                    // output rows per 128-row half
  int win_half_rows;               // shared-memory rows per half = win_rows * win_pitch
  int win_box_rows;                // input rows per box = m_halves * win_rows + R - 1
  int win_row_blocks;              // tiles per image = ceil(Ho / (m_halves * win_rows))
  int win_R, win_S;                // filter extent
  int win_pad_h, win_pad_w;
  uint32_t win_stage_bytes;        // A stage size (box plus the rows junk MMA rows may read)

  // Gather A loader (forward convs whose channel rows TMA cannot address:
  // C_in * elt not a multiple of 16 bytes, or under 32).  An A row is laid
  // out as R runs; run r holds the input bytes under filter row r and taps
  // s = 0 .. S-1, all channels: with dil_w = 1 these are S adjacent pixels,
  // i.e. g_run_len_bytes contiguous bytes of the NHWC input.  Each run is
  // zero-padded to g_run_bytes (a multiple of 16) so every 16-byte piece of
  // an A row comes from one input address.  The producer warps build A with
  // plain loads and shared-memory stores.
  int gather;
  const uint8_t* g_input;
  long long g_input_bytes;
  int g_n, g_h, g_w, g_c;          // input shape (NHWC)
  int g_elt;                       // bytes per element
  int g_runs;                      // runs per A row (= R)
  int g_s;                         // filter extent along S
  int g_run_len_bytes;             // valid bytes of a run (S * C_in * elt)
  int g_run_bytes;                 // padded bytes of a run
  // Row staging (when an input row, W * C_in * elt bytes, is a multiple of 16
  // bytes): the input rows a tile reads arrive in shared memory by bulk
  // copies, one tile ahead, and the pieces are cut from there.  Slot j of a
  // tile's buffer holds padded input row g_first + j, where padded row
  // g = n * g_pr + (iy + pad_h) enumerates each image's rows oy*stride +
  // r*dil_h; slots in the padding stay unloaded.
  // A slot is [g_slot_pad zero bytes][the row][zero bytes], g_slot_bytes in
  // all: reads of pixels left or right of the image see zeros.
  int g_stage;
  int g_slots;                     // slots per staging buffer
  int g_slot_bytes;                // slot stride (multiple of 16)
  int g_slot_pad;                  // zero bytes before the row (multiple of 16)
  int g_row_bytes;                 // W * C_in * elt
  int g_pr;                        // padded rows per image: (Ho-1)*stride_h + (R-1)*dil_h + 1
  FastDiv g_div_run, g_div_pr;     // division by g_run_bytes and by g_pr
  uint32_t g_stage_bytes;          // bytes per staging buffer

  // Stream-K (convs whose tiles fill less than one wave of CTAs): the
  // sequence of (tile, k-block) iterations, tile by tile, is cut into equal
  // contiguous shares, one per CTA, and each share into work items at tile
  // boundaries.  A CTA whose share starts inside a tile writes that item's
  // fp32 accumulators to its partial slot and raises its epilogue warps'
  // flags to sk_epoch; the CTA holding the tile's first k-block adds every
  // such partial and runs the epilogue.
  int streamk;
  long long sk_iters;                    // iterations in all (< 2^31)
  long long sk_iter_start[kMaxPhases + 1];  // first iteration of each phase
  int sk_kpt[kMaxPhases];                // k-blocks per tile of each phase (> 0)
  FastDiv sk_div_kpt[kMaxPhases];
  uint32_t sk_epoch;                     // this launch's flag value (never 0)
  unsigned int* sk_flags;                // [CTA][epilogue warp]
  float* sk_partials;                    // [CTA][m_halves * bn / 16][128 rows][16]
  uint32_t sk_slot_floats;               // floats per CTA slot

  int epi_mode;                    // 0 direct stores, 1 TMA store [M][C_out], 2 TMA 4-D phase grid,
                                   // 3 TMA 4-D row window
  int cw;                          // epilogue chunk width in columns (16, 32 or 64)
  int src_bufs;                    // residual-source tile buffers (0, 1 or 2)
  uint32_t src_chunk_bytes;        // stride of one (half, chunk) item in a source buffer
  int valid_rows;                  // TMEM lanes per half that map to stored rows (128, or win_half_rows)
  int stg_bufs;                    // output staging buffers per epilogue group (0: in place)

  int Ho, Wo, Cout;
  int vec_ok;                      // C_out * 2 bytes is a multiple of 16: 16-B stores
  // Direct epilogue of few output channels (C_out <= 16, not a multiple of
  // 8; one phase, one group, rows contiguous in the output): each epilogue
  // warp assembles its 32 rows' outputs in a shared-memory stage and writes
  // them as 16-byte words (seg_slot_bytes per stage; an output and a source
  // stage per warp of the first epilogue group, from off_seg).
  int seg_store;
  uint32_t off_seg;
  uint32_t seg_slot_bytes;
  int has_residual;
  int epilogue;
  float beta;
  const void* src;
  void* out;
  unsigned int* status;
  long long timeout_cycles;        // limit of every bounded wait, in SM cycles
  uint32_t wait_hint_ns;           // suspend hint for waits off the MMA's critical path (0: poll)
  int fault_mode;                  // test hook: 1 = CTA 0 skips its first arrive;
                                   // 2 = stream-K partials never raise their flags
};

}  // namespace convgb300
