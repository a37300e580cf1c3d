// pod_internal.h — definitions shared by the host planner (planner.cpp) and the CUDA
// translation unit (pod_attn.cu): the work-item encoding, the workspace layout and the tile
// constants. Plain C++ (no CUDA headers) so the planner compiles with g++ alone.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/pod_attn.h"

namespace pod {

// Shape constants of this build (the library rejects other shapes with UNSUPPORTED).
constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;          // tokens per paged K/V block
constexpr int kMaxGroup = 8;            // query heads per KV head handled by the decode path

// Prefill tile: 128 query rows x 64 keys per step; QKᵀ and PV on the tcgen05 tensor cores.
constexpr int kTileM = 128;
constexpr int kTileN = 64;
constexpr int kKStages = 3;             // K tiles in flight (needed first, by S = Q·Kᵀ)
constexpr int kVStages = 2;             // V tiles in flight (needed a softmax later, by P·V)

// One CTA shape serves both item kinds ("POD-Attention" digest, §"가상 CTA와 SM별 균형": one
// shared-memory configuration for both operations).
constexpr int kThreads = 192;           // 6 warps
constexpr int kWarps = kThreads / 32;
constexpr int kDecodeSlots = 2;         // K+V blocks in flight per decode warp

// Shared-memory map (bytes from the dynamic shared-memory base, which the hardware places at
// a 1024-byte boundary; the kernel checks this and reports an error otherwise).
constexpr int kSmemQ = kTileM * kHeadDim * 2;                  // 32 KiB
constexpr int kSmemKTile = kTileN * kHeadDim * 2;              // 16 KiB (K or V tile)
constexpr int kSmemUnion = kSmemQ + (kKStages + kVStages) * kSmemKTile;  // 112 KiB
constexpr int kSmemDecodeSlot = 2 * kBlockSize * kHeadDim * 2; // 8 KiB (K block + V block)
constexpr int kSmemDecodeRing = kWarps * kDecodeSlots * kSmemDecodeSlot;  // 96 KiB
constexpr int kSmemScores = kWarps * kMaxGroup * kBlockSize * 4;   // per-warp p exchange
static_assert(kSmemDecodeRing + kSmemScores <= kSmemUnion, "decode ring too big");
constexpr int kSmemBarriers = 256;                                   // mbarriers + scalars
constexpr int kSmemTotal = kSmemUnion + kSmemBarriers;
// Two CTAs per SM: 2 x (kSmemTotal + 1 KiB the driver reserves per CTA) <= 228 KiB.
static_assert(2 * (kSmemTotal + 1024) <= 228 * 1024, "two CTAs per SM must fit");

// TMEM columns per CTA: O (128 fp32 columns) + two S buffers of 64 columns. Two CTAs per SM
// fit the 512 columns of an SM.
constexpr int kTmemCols = 256;
constexpr int kTmemO = 0;
constexpr int kTmemS0 = 128;

// Work item: kItemWords int32 words.
//   [0] kind         0 = prefill, 1 = decode
//   [1] seq          prefill: chunk index s in [0, Np); decode: d in [0, Nd)
//   [2] tile / kvh   prefill: 128-row query tile index t; decode: kv-head g
//   [3] head         prefill: query head h; decode: 0
//   [4] key_begin    first key row of this split (prefill: multiple of 64; decode: of 16)
//   [5] key_end      one past the last key row this split may read
//   [6] unit         -1 = the only split (write the output directly), else the unit index
//   [7] split        split index within the unit
constexpr int kItemWords = 8;
// Unit (an output assembled from several splits): kUnitWords int32 words.
//   [0] nsplit  [1] first partial slot  [2] kind  [3] unused
constexpr int kUnitWords = 4;

// Partial-result slots: fp32 o[rows][128] then m[rows] then l[rows] (m, l in log2 units).
constexpr int kPrefillSlotFloats = kTileM * (kHeadDim + 2);
#ifdef __CUDACC__
__host__ __device__
#endif
inline int decode_slot_floats(int group) { return group * (kHeadDim + 2); }

// Counter block of one launch mode (fused, prefill-only, decode-only), int32 words:
//   [0] prefill ticket  [1] decode ticket  [2] exited CTAs  [3] unused
//   [4 .. 4+num_sms)    prefill items running on each SM
constexpr int kCounterHeader = 4;

enum LaunchMode { kModeFused = 0, kModePrefillOnly = 1, kModeDecodeOnly = 2 };

// Workspace layout (byte offsets, each 256-aligned).
struct WorkspaceLayout {
  size_t status = 0;        // int32 status word, int32 abort word
  size_t counters = 0;      // 3 counter blocks
  size_t counter_block_words = 0;
  size_t arrive = 0;        // int32 per unit
  size_t items_p = 0;       // prefill items
  size_t items_d = 0;       // decode items
  size_t units = 0;         // unit table
  size_t partial_p = 0;     // prefill partial slots
  size_t partial_d = 0;     // decode partial slots
  size_t records = 0;       // instrumentation records (0 bytes when off)
  size_t zero_bytes = 0;    // bytes from 0 that pod_attn_upload clears (status..arrive end)
  size_t total = 0;
};

}  // namespace pod

// The opaque plan.
struct pod_attn_plan_s {
  pod_attn_problem prob{};
  pod_attn_options opt{};
  int group = 1;
  int num_sms = 0, ctas_per_sm = 2, max_prefill_per_sm = 1;
  int grid_fused = 0, grid_prefill = 0, grid_decode = 0;
  std::vector<int32_t> cu, kv;            // host copies of the lengths
  std::vector<int32_t> items_p, items_d;  // kItemWords each
  std::vector<int32_t> units;             // kUnitWords each
  int num_p_slots = 0, num_d_slots = 0;
  pod::WorkspaceLayout ws;
  double est_prefill_flops = 0, est_prefill_bytes = 0, est_decode_bytes = 0,
         est_decode_flops = 0;
  // CUDA-side state owned by pod_attn.cu (events for the STREAMS variant, cached tensor maps).
  void* cuda_state = nullptr;
};

namespace pod {
// Planner entry (planner.cpp). Fills everything but cuda_state. num_sms must be > 0.
pod_attn_status build_plan(const pod_attn_problem& prob, const int32_t* cu, const int32_t* kv,
                           const pod_attn_options& opt, int num_sms, pod_attn_plan_s* plan);
}  // namespace pod
