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

// One persistent CTA per SM holds two concurrent virtual-CTA slots ("POD-Attention" digest,
// §"가상 CTA와 SM별 균형": prefill and decode work placed side by side on every SM):
//  * the prefill slot (warps 0-11): one pipeline over the SM's TMEM that runs a 128-row query
//    tile against a range of K/V tiles — warps 0 and 2 issue the TMA loads (K and V) of one
//    ring of K and V tiles, warps 1 and 3 issue the P·V and the S tcgen05 MMAs, and warps 4-11 load the tile's
//    queries into TMEM and run the softmax, two threads per query row (warps w and w + 4
//    share the row's TMEM lane, each takes 64 of a step's 128 keys);
//  * the decode slot (warps 12-15): decode items, on their own ticket loop.
// Once the prefill list is drained, the prefill slot's warps 4-7 and 8-11 become two more
// 4-warp decode slots. Every decode item thus runs on exactly 4 warps, whichever slot takes it,
// so its arithmetic (and result) does not depend on where it ran.
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPrefillThreads = 384;    // warps 0-11
constexpr int kSoftmaxWarp0 = 4;        // first softmax warp (keys 0-63: 4-7, 64-127: 8-11)
constexpr int kDecodeWarp0 = 12;        // decode slot: warps 12-15
constexpr int kDecodeWarps = 4;
constexpr int kDecodeSlots = 2;         // K+V blocks in flight per decode warp (bf16 cache)
constexpr int kDecodeSlotsFp8 = 3;      // ... on the e4m3 cache (half the bytes per block)

// Prefill tile: 128 query rows = T tokens x hp query heads of one kv-head group (hp = the largest
// power of two dividing the group size, T = 128 / hp; row r is token r / hp, head h0 + r % hp).
// All hp heads read the same K and V, so one K/V tile serves hp heads ("LLMSO - W4", §"KV 헤드
// 줄이기": the heads of a group share their K/V).
// Prefill item: one tile (tokens tT .. tT+T-1 of one chunk, one head block) against a range of
// keys. Prefill step: the tile x 128 keys. The tile has two S buffers in TMEM (step n uses
// buffer n & 1), so S of the next step is computed while the softmax of this one runs, and its
// queries sit in TMEM as the A operand of the S MMAs, so the tensor cores read only K and V from
// shared memory. K and V tiles share one ring of kKVStages tiles, loaded in the order the MMAs
// consume them: K(0), K(1), then V(j), K(j + 2) for each step j.
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kKVStages = 5;

// Shared-memory map (bytes from the dynamic shared-memory base, which the hardware places at
// a 1024-byte boundary; the kernel checks this and reports an error otherwise).
constexpr int kSmemKTile = kTileN * kHeadDim * 2;                  // 32 KiB (K or V tile)
constexpr int kSmemPrefill = kKVStages * kSmemKTile;               // 160 KiB
constexpr int kSmemDecodeSlot = 2 * kBlockSize * kHeadDim * 2;     // 8 KiB (K block + V block)
constexpr int kSmemDecodeRing = kDecodeWarps * kDecodeSlots * kSmemDecodeSlot;  // 64 KiB
constexpr int kSmemScoresPerWarp = kMaxGroup * kBlockSize * 4;     // p exchange of one warp
constexpr int kSmemDecodeOff = kSmemPrefill;                       // decode slot's region
constexpr int kSmemScoresOff = kSmemDecodeOff + kSmemDecodeRing;   // its score exchange
constexpr int kSmemCtlOff = kSmemScoresOff + kDecodeWarps * kSmemScoresPerWarp;
constexpr int kSmemBarriers = 1024;                                 // mbarriers + scalars
constexpr int kSmemTotal = kSmemCtlOff + kSmemBarriers;
static_assert(kSmemTotal <= 227 * 1024, "one CTA per SM must fit");
// the prefill slot's region also serves as the rings and score areas of its two decode slots
static_assert(2 * (kSmemDecodeRing + kDecodeWarps * kSmemScoresPerWarp) <= kSmemPrefill,
              "the two decode slots of the prefill warps must fit the prefill region");

// TMEM columns (the whole SM; lane r is tile row r): the O accumulator (fp32, 128 columns), two
// S buffers (fp32, 128 columns each), the tile's queries (bf16 pairs, 64 columns: column c holds
// dims 2c and 2c + 1) and a few columns through which the two softmax threads of a row exchange
// their max and sum. A step's softmax writes its P (bf16 pairs, 128 keys) over the first 64
// columns of its S buffer; S of step n + 2 is issued into that buffer once the P·V(n) that reads
// P has completed.
constexpr int kTmemCols = 512;
constexpr int kTmemO = 0;
constexpr int kTmemS = 128;    // + 128 * (step & 1)
constexpr int kTmemQ = 384;
constexpr int kTmemX = 448;    // [0, 4): maxima by step parity and half; [4, 6): sums by half

// Work item: kItemWords int32 words.
//   [0] kind         0 = prefill, 1 = decode
//   [1] seq          prefill: chunk index s in [0, Np); decode: d in [0, Nd)
//   [2] tile / kvh   prefill: index t of the tile (chunk tokens Tt .. Tt + T - 1, with
//                    T = 128 / hp tokens per tile); decode: kv-head g
//   [3] head         prefill: first query head h0 of the tile's hp heads; decode: 0
//   [4] key_begin    first key row of this split (prefill: multiple of 128; decode: of 16)
//   [5] key_end      one past the last key row this split may read
//   [6] unit         -1 = the only split (write the output directly), else the unit index
//   [7] split        split index within the unit
constexpr int kItemWords = 8;
// Unit (an output assembled from several splits): kUnitWords int32 words.
//   [0] nsplit  [1] first partial slot  [2] kind  [3] unused
constexpr int kUnitWords = 4;

// Most splits of one prefill output (the planner's cap; the merge keeps one weight per split).
constexpr int kMaxPrefillSplits = 8;
// Most splits of one decode output (the planner's cap; the merge keeps G weights per split in
// shared memory).
constexpr int kMaxDecodeSplits = 64;

// Partial-result slots. A prefill slot holds the 128 rows of a tile: O / l as bf16 [rows][128]
// (in 8-column chunks interleaved across each 32 rows), then fp32 m[rows] and l[rows] (m in
// log2 units). A decode slot: fp32 o[rows][128] then m[rows], l[rows].
constexpr int kPrefillSlotBytes = kTileM * kHeadDim * 2 + 2 * kTileM * 4;
#ifdef __CUDACC__
__host__ __device__
#endif
inline int decode_slot_floats(int group) { return group * (kHeadDim + 2); }

// Counter block of one launch mode (fused, prefill-only, decode-only, append-only), int32 words:
//   [0] prefill ticket  [1] decode ticket  [2] exited CTAs
//   [3] CTAs that have finished their share of the KV append (pod_attn_run_append)
//   [4 .. 4+num_sms)    decode items the prefill slot of each SM has taken (diagnostics)
constexpr int kCounterHeader = 4;

enum LaunchMode { kModeFused = 0, kModePrefillOnly = 1, kModeDecodeOnly = 2, kModeAppendOnly = 3 };
constexpr int kNumModes = 4;

// Workspace layout (byte offsets, each 256-aligned).
struct WorkspaceLayout {
  size_t status = 0;        // int32 status word, int32 abort word
  size_t counters = 0;      // kNumModes counter blocks
  size_t counter_block_words = 0;
  size_t arrive = 0;        // int32 per unit
  size_t items_p = 0;       // prefill items
  size_t items_d = 0;       // decode items
  size_t units = 0;         // unit table
  size_t new_rows = 0;      // (sequence, position) of each appended token (KV append)
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
  int head_pack = 1;                      // hp: query heads per prefill tile
  int tile_tokens = pod::kTileM;          // T = 128 / hp: tokens per prefill tile
  int num_sms = 0, ctas_per_sm = 1;
  int max_prefill_ctas = 0;               // CTAs whose prefill slot takes prefill items (CTAs 0..)
  int grid_fused = 0, grid_prefill = 0, grid_decode = 0;
  std::vector<int32_t> cu, kv;            // host copies of the lengths
  std::vector<int32_t> items_p, items_d;  // kItemWords each
  std::vector<int32_t> units;             // kUnitWords each
  std::vector<int32_t> new_rows;          // 2 words per new token: prefill chunk tokens in
                                          // order, then one per decode sequence
  int num_p_slots = 0, num_d_slots = 0;
  pod::WorkspaceLayout ws;
  // Bytes [0, ws.partial_p) of the workspace as pod_attn_upload writes them: the zeroed status,
  // counters and arrival counters, then the work lists at their offsets (one host-to-device
  // copy per upload).
  std::vector<uint8_t> upload_image;
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
