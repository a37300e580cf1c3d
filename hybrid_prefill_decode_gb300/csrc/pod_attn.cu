// pod_attn.cu — GB300 (sm_103a) kernels and C ABI of hybrid prefill+decode attention.
//
// One persistent kernel runs two kinds of virtual CTAs ("POD-Attention" digest, Silicon &
// Systems, §"동시 실행만으로 부족한 이유" and §"가상 CTA와 SM별 균형"):
//
//  * prefill item — two 128-row query tiles (each 128/hp tokens x hp heads of one kv-head
//    group) of one chunk against a range of keys: S = Q·Kᵀ and O += P·V on the tcgen05 tensor
//    cores with S and O in TMEM, Q/K/V staged by TMA through the paged block table, causal mask
//    and online softmax (running max m and sum l, rescale by 2^(m_old - m_new); "Week 6: Beyond
//    PyTorch: Custom Kernel과 vLLM", §"FlashAttention의 single-pass 트릭"; "LLMSO - W4",
//    §"FlashAttention — I/O를 줄이는 방향"). Warp 0 issues TMA (Q, then K and V through one
//    ring), warp 1 issues the S MMAs and warp 3 the P·V MMAs of both tiles, and two warpgroups
//    (4-7, 8-11) do the softmax of tile A and tile B, one query row per thread, so one tile's
//    softmax runs while the tensor cores work on the other tile.
//  * decode item — one sequence, one kv-head with its G query heads, a range of 16-row paged
//    blocks: each warp streams its blocks into a private two-slot shared-memory ring (4 KiB bulk
//    copies for MHA, TMA boxes for GQA), keeps an online softmax per head, and reduces q·k with
//    warp shuffles (MHA) or warp-level MMAs over the G heads (GQA) ("LLMSO - W4",
//    §"FlashDecoding — decode 단계의 병렬성 확보", §"KV 헤드 줄이기"). Over an e4m3 cache
//    (pod_attn_run_decode_fp8) every group size runs on f16 warp MMAs.
//
// One hardware CTA per SM runs a prefill slot and a decode slot side by side, each pulling
// tickets from its own list, so both kinds share every SM (§"가상 CTA와 SM별 균형"); %smid is
// recorded per item. Outputs split along the keys are merged exactly
// by log-sum-exp by whichever split finishes last (no CTA ever waits for another CTA, so the two
// kinds cannot deadlock; §"가상 CTA와 SM별 균형": exact synchronisation where partials meet).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "pod_internal.h"
#include "ptx.cuh"

namespace pod {

using namespace ptx;

constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s: no healthy wait comes close
// Longest hardware sleep of one poll for roles off the softmax's critical path; a completed
// phase wakes the thread earlier.
constexpr uint32_t kSleepNs = 20000;

struct Params {
  const uint16_t* q_prefill;
  const uint16_t* q_decode;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* block_tables;
  const int32_t* cu_seqlens;
  const int32_t* kv_lens;
  uint16_t* o_prefill;
  uint16_t* o_decode;
  const int32_t* items_p;
  const int32_t* items_d;
  const int32_t* units;
  float* partial_p;
  float* partial_d;
  int32_t* counters;  // this launch mode's counter block
  int32_t* arrive;
  int32_t* status;    // [0] status word, [1] unused
  pod_attn_item_record* records;
  // KV append (pod_attn_run_append): the new K/V rows and where they go
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool_w;
  uint16_t* v_pool_w;
  const int32_t* new_rows;  // (sequence, position) per new token
  int32_t n_new;            // new tokens this launch appends (0 = no append)
  int32_t new_first;        // index of the first of them in k_new / v_new / new_rows
  int32_t wait_append;      // items wait until every CTA has done its share of the append
  // FP8 cache (pod_attn_run_decode_fp8): e4m3 pools, K scale per (kv-head, channel), V scale
  // per (block, kv-head, row)
  const uint8_t* k8;
  const uint8_t* v8;
  const float* k_scale;
  const float* v_scale;
  int32_t n_items_p, n_items_d;
  int32_t Hq, Hkv, G, Np, Nd, num_blocks, maxb;
  int32_t pool_rows;  // num_blocks * Hkv * 16: first row past the pools (TMA fills zeros)
  int32_t num_sms;
  int32_t max_prefill_ctas;  // CTAs 0 .. max_prefill_ctas - 1 take prefill items
  int32_t hp_log2;    // prefill tile: 2^hp_log2 heads x tq tokens
  int32_t causal;     // 0: chunk tokens see every row of their sequence
  int32_t head_dim;   // 128 or 64 (selects the kernel instantiation)
  int32_t tq;
  int32_t mode;
  float scale_log2;   // scale * log2(e): scores are kept in base-2 units
  uint64_t timeout_ns;
};

struct SmemCtl {
  uint64_t q_full;                 // the item's queries are in TMEM (one arrival per warp)
  uint64_t kv_full[kKVStages];     // the ring stage holds its K or V tile
  uint64_t kv_empty[kKVStages];    // the MMAs that read the stage completed
  uint64_t s_full[2];              // [buffer] S of the buffer's step computed
  uint64_t p_ready[2];             // [buffer] P of the step written (one arrival per warp)
  uint64_t pv_done;                // one completion per step: its P·V completed
  uint64_t o_done;                 // the item's last P·V completed
  uint64_t dslot[kWarps][kDecodeSlotsFp8];  // decode rings, by absolute warp (slots in use:
                                            // kDecodeSlots on a bf16 cache, kDecodeSlotsFp8 on e4m3)
  uint32_t tmem_base;
  int abort;
  int item_kind[5];                // per slot: 0 = prefill, 1 = decode, 2-3 = the prefill slot's
  int item_idx[5];                 //   warps 4-7 / 8-11 once prefill work is drained, 4 = its
  int merge_last[5];               //   warps 0-3 (FP8 cache decode only)
};
static_assert(sizeof(SmemCtl) <= kSmemBarriers, "control block too big");

// Pipeline positions; each role advances the fields it owns, across items.
struct PipeState {
  uint32_t q_cnt = 0;   // prefill items (query-tile loads)
  bool appended = false;  // this thread has seen the launch's KV append complete
  uint32_t t_cnt = 0;   // 128-key steps (K/V ring entries 2n, 2n + 1; S and P barriers)
  uint32_t dphase = 0;  // decode ring: one parity bit per slot of this warp
};

// Where a decode item runs: `nw` (= 4) warps from absolute warp `w0`, their rings and score
// areas, the named barrier of the slot that runs it and the slot's index in the control block.
struct DecodeCtx {
  int w0, nw;
  uint8_t* ring;        // nw * kDecodeSlots * kSmemDecodeSlot bytes; also the combine scratch
  float* scores;        // nw * kMaxGroup * kBlockSize floats
  int bar_id, bar_threads, first_thread, slot;
};

constexpr uint32_t kIdescS = idesc_bf16(kTileM, kTileN, 0, 0);     // S = Q Kᵀ, both K-major

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return static_cast<uint16_t>(pack_bf16x2(f, 0.f) & 0xFFFFu);
}

// ============================================================================ KV append
// The step before attention ("Week 6: Beyond PyTorch: Custom Kernel과 vLLM", §"PagedAttention":
// the cache is append-only; §"한 스텝에 여러 종류의 request 섞기"): every new token's K and V row
// of each kv-head is written into its paged block. One warp per (token, kv-head): lanes 0-15 copy
// the K row, lanes 16-31 the V row, 16 bytes each (coalesced 256-byte rows).
template <int HD>
__device__ void append_rows(const Params& p) {
  constexpr int kVec = HD / 8;  // 16-byte vectors per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.n_new * p.Hkv;
  for (int u = blockIdx.x * kWarps + warp; u < units; u += gridDim.x * kWarps) {
    const int tok = p.new_first + u / p.Hkv, g = u % p.Hkv;
    const int seq = p.new_rows[2 * tok], pos = p.new_rows[2 * tok + 1];
    const int phys = p.block_tables[(size_t)seq * p.maxb + pos / kBlockSize];
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) record_error(p.status, POD_ATTN_ERR_BAD_INDEX);
      continue;
    }
    const size_t row = ((size_t)phys * p.Hkv + g) * kBlockSize + pos % kBlockSize;
    if (lane >= 2 * kVec) continue;  // lanes [0, kVec) copy the K row, [kVec, 2 kVec) the V row
    const bool is_k = lane < kVec;
    const int v = lane % kVec;
    const uint16_t* src = (is_k ? p.k_new : p.v_new) + ((size_t)tok * p.Hkv + g) * HD;
    uint16_t* dst = (is_k ? p.k_pool_w : p.v_pool_w) + row * HD;
    reinterpret_cast<uint4*>(dst)[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
  }
}

// Before a thread issues copies of pool rows that the launch appends: wait (bounded) until every
// CTA has finished its share, then order those generic-proxy writes before this thread's
// async-proxy (TMA, bulk copy) reads. Returns false on timeout or abort.
__device__ bool wait_appended(const Params& p, PipeState& ps, const WaitCtx& wc) {
  if (!p.wait_append || ps.appended) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    int done;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(done) : "l"(p.counters + 3) : "memory");
    if (done >= (int)gridDim.x) break;
    if (*wc.abort) return false;
    if (globaltimer() - t0 > wc.timeout_ns) {
      *wc.abort = 1;
      record_error(wc.status, POD_ATTN_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  ps.appended = true;
  return true;
}

// ============================================================================ prefill item
// One prefill item: one 128-row query tile of one chunk and head block against a range of keys
// in 128-key steps (the single-pass online softmax of "Week 6: Beyond PyTorch: Custom Kernel과
// vLLM", §"FlashAttention의 single-pass 트릭"; "LLMSO - W4", §"FlashAttention — I/O를 줄이는
// 방향"). Steps are numbered n by a counter that runs on across items. TMEM holds the tile's O
// accumulator, two S buffers (step n uses buffer n & 1) and the tile's queries, which are the A
// operand of every S MMA: S(j + 1) is computed while the softmax of step j runs, and the tensor
// cores read only K and V from shared memory.
//  * Warps 0 (K) and 2 (V) load K and V through one ring of kKVStages tiles in the order the
//    MMAs consume them: K(0), K(1), then V(j) and K(j + 2) for each step j.
//  * Warp 1 issues the P·V MMAs, P·V(j) once P(j) is written; warp 3 issues the S MMAs: S(0),
//    S(1), then S(j + 2) into the S buffer whose P P·V(j) reads, once P·V(j) has completed.
//  * Warps 4-11 load the tile's queries into TMEM and run the softmax, two threads per query
//    row: warps w and w + 4 reach the same TMEM lanes (rows) and take keys 0-63 and 64-127 of
//    each step. The two halves of a row exchange their maxima through TMEM, so that P of the
//    whole row is taken against one max; each half keeps its own share of the row sum l.
// Each row keeps its running max m (log2 units); O is rescaled only when the row's max grows by
// more than 2^8 (the lazy-rescale threshold), once the previous P·V has completed; the epilogue
// divides by l. HD (head dim) is 128 or 64; a 64-dim head uses the first half of every K/V tile
// and of O.
template <int HD>
__device__ void prefill_item(const Params& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                             const CUtensorMap* tmkb, const CUtensorMap* tmvb,
                             const int32_t* it, uint8_t* smem, SmemCtl* ctl, PipeState& ps,
                             const WaitCtx& wc) {
  static_assert(HD == 64 || HD == 128, "head dim");
  constexpr int kHalves = HD / 64;                  // 64-dim halves (128-byte swizzle atoms)
  constexpr uint32_t kIdescPV = idesc_bf16(kTileM, HD, 0, 1);  // O += P V, V N-major
  constexpr uint32_t kTileBytes = kTileN * HD * 2;
  constexpr uint32_t kBlockBytes = kBlockSize * HD * 2;
  constexpr int kBlocksPerTile = kTileN / kBlockSize;  // 8
  // K and V tiles are laid out block by block, so that one box of a per-block map brings all of
  // a paged block (the TMA unit takes ~60 cycles per box, whatever its size):
  //  * V: [block][64-dim half][16 rows][128 bytes]; each P·V MMA reads one block;
  //  * K (head dim 128): [block][8-row group][64-dim half][8 rows][128 bytes], so that the 8-row
  //    groups of one half lie 2 KiB apart throughout the tile and an S MMA reads 16 dims of all
  //    128 keys with one descriptor (stride 2 KiB, the second half 1 KiB further on); with head
  //    dim 64 a block is [16 rows][128 bytes] and the groups lie 1 KiB apart.
  constexpr uint32_t kVBlockBytes = kBlockBytes;      // 4 KiB (head dim 128) or 2 KiB (64)
  constexpr uint32_t kKGroupStride = HD == 128 ? 2048 : 1024;  // 8-row groups of one K half
  constexpr uint32_t kKHalfOff = 1024;                // second 64-dim half of a K group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = it[1], t = it[2], h0 = it[3], kb = it[4], ke = it[5], unit = it[6], split = it[7];
  const int g = h0 / p.G;  // the tile's heads h0 .. h0 + hp - 1 share kv-head g
  const int q0 = p.cu_seqlens[s];
  const int qlen = p.cu_seqlens[s + 1] - q0;
  const int L = p.kv_lens[s];
  const int P = L - qlen;  // cached prefix rows before this chunk
  const int ntiles = (ke - kb + kTileN - 1) / kTileN;  // >= 1 (every item has keys)
  const uint32_t n0 = ps.t_cnt;  // this item's first step
  const uint32_t sRing = smem_u32(smem);
  // The item's 2 ntiles ring entries in consumption order: K(0), K(1), then V(j), K(j + 2) for
  // j < ntiles - 2, then the last two V. Entry ei is ring entry 2 n0 + ei overall (stage
  // (2 n0 + ei) % kKVStages).
  auto ek = [&](int i) { return i < 2 ? i : 2 * i - 1; };              // entry of K(i)
  auto ev = [&](int j) { return j < ntiles - 2 ? 2 + 2 * j : ntiles + j; };  // entry of V(j)
  auto stage_of = [&](int ei) { return (2 * n0 + (uint32_t)ei) % kKVStages; };
  auto phase_of = [&](int ei) { return ((2 * n0 + (uint32_t)ei) / kKVStages) & 1u; };

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 0 loads the K entries and warp 2 the V entries (a warp issues about one box per 100
    // cycles, and a step needs 16). Lane i holds the block-table entry of block i of the next 4
    // steps (32 blocks): one coalesced read instead of a dependent global read per block. A stage
    // is free once the MMAs that read it completed (kv_empty: one commit after them).
    const int my_kv = warp == 2;
    const int32_t* bt_row = p.block_tables + (size_t)s * p.maxb;
    const int nblk_item = (ke - kb + kBlockSize - 1) / kBlockSize;
    const int blk0 = kb / kBlockSize;
    auto bt_fetch = [&](int j4) -> int {  // entries of steps j4 .. j4 + 3
      const int bi = j4 * kBlocksPerTile + lane;
      return bi < nblk_item ? bt_row[blk0 + bi] : -1;
    };
    // Each stream (K, V) keeps its own window of block-table entries (the one of its current 4
    // steps and the next); each stream reads its steps in order.
    int cur_k = -1, nxt_k = bt_fetch(0), win_k = -1;
    int cur_v = -1, nxt_v = nxt_k, win_v = -1;
    auto advance = [&](int& cur, int& nxt, int& win, int j) {
      const int w = j >> 2;
      if (w == win) return;
      win = w;
      const bool in_range = w * 4 * kBlocksPerTile + lane < nblk_item;
      cur = nxt;
      if ((w + 1) * 4 < ntiles) nxt = bt_fetch((w + 1) * 4);
      if (in_range && (cur < 0 || cur >= p.num_blocks)) {
        record_error(p.status, POD_ATTN_ERR_BAD_INDEX);
        cur = 0;
      }
      if (!in_range) cur = -1;
    };
    // Rows past the sequence end inside its last block may hold anything (even NaN); P is zero
    // there but 0 * NaN is not. So when the item reads that block, this warp writes its V rows
    // itself (the valid rows, then zeros) in the layout TMA's 128-byte swizzle gives.
    const int tail_blk = ((L & 15) && ke > (L & ~15)) ? L / kBlockSize - blk0 : -1;
    // the chunk's own rows [P, P + qlen) may be appended by this launch
    int oka = 1;
    if (lane == 0 && ke > P) oka = wait_appended(p, ps, wc);
    for (int ei = 0; __shfl_sync(0xffffffffu, oka, 0) && ei < 2 * ntiles; ++ei) {
      // which tile entry ei brings (the inverse of ek / ev above)
      int kv, j;
      if (ntiles == 1) {
        kv = ei, j = 0;
      } else if (ei < 2) {
        kv = 0, j = ei;
      } else if (ei - 2 < 2 * (ntiles - 2)) {
        const int r = ei - 2;
        kv = (r & 1) ? 0 : 1;
        j = (r & 1) ? (r >> 1) + 2 : r >> 1;
      } else {
        kv = 1, j = ei - ntiles;
      }
      if (kv != my_kv) continue;
      if (kv) advance(cur_v, nxt_v, win_v, j);
      else advance(cur_k, nxt_k, win_k, j);
      const int cur = kv ? cur_v : cur_k;
      // lane i copies block i of the tile (all of its dims in one box); one warp instruction
      // issues all the copies
      const int bl = lane % kBlocksPerTile;
      const int el = __shfl_sync(0xffffffffu, cur, (j & 3) * kBlocksPerTile + bl);
      const int yl = el < 0 ? p.pool_rows : (el * p.Hkv + g) * kBlockSize;  // past the pool: zeros
      const uint32_t stage = stage_of(ei);
      int w = 1;
      // the stage's previous use has completed (a fresh barrier passes); polled without a
      // sleep hint, as a stage often frees while the next load is already due
      if (lane == 0) w = mbar_wait(smem_u32(&ctl->kv_empty[stage]), phase_of(ei) ^ 1u, wc);
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      const uint32_t dst = sRing + stage * kSmemKTile;
      const int tb = kv == 1 ? tail_blk - j * kBlocksPerTile : -1;
      const bool tail = tb >= 0 && tb < kBlocksPerTile;  // V's partly filled block is here
      if (tail) {
        const int r = L & 15;
        const int yt = __shfl_sync(0xffffffffu, yl, tb);  // the block's first row
        const uint16_t* src = p.v_pool + (size_t)yt * HD;
        uint8_t* base = smem + (dst - sRing) + tb * kVBlockBytes;
#pragma unroll
        for (int c = lane; c < kBlockSize * 8 * kHalves; c += 32) {  // 16-byte chunks
          const int i = c / (8 * kHalves), hf = (c >> 3) % kHalves, q16 = c & 7;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (i < r) v = __ldcg(reinterpret_cast<const uint4*>(src + (size_t)i * HD + hf * 64) + q16);
          *reinterpret_cast<uint4*>(base + hf * 2048 + i * 128 + ((q16 ^ (i & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint32_t full = smem_u32(&ctl->kv_full[stage]);
      if (lane == 0) mbar_arrive_expect_tx(full, tail ? kTileBytes - kBlockBytes : kTileBytes);
      __syncwarp();
      if (kv == 0) {
        if (lane < kBlocksPerTile) {
          // head dim 128: box {64 dims, 8 rows, 2 halves, 2 row groups}; 64: {64 dims, 16 rows}
          if constexpr (HD == 128) tma_load_4d(dst + bl * kBlockBytes, tmkb, full, 0, 0, 0, yl / 8);
          else tma_load_2d(dst + bl * kBlockBytes, tmk, full, 0, yl);
        }
      } else if (lane < kBlocksPerTile && !(tail && bl == tb)) {
        if constexpr (HD == 128) tma_load_3d(dst + bl * kVBlockBytes, tmvb, full, 0, yl, 0);
        else tma_load_2d(dst + bl * kVBlockBytes, tmv, full, 0, yl);
      }
      __syncwarp();
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 1 issues the P·V MMAs and warp 3 the S MMAs: the tensor cores queue only a couple of
    // MMAs, so one thread that waits on a barrier between its batches leaves them idle, while
    // two threads keep them fed. S(j + 2) overwrites P(j), so it is issued once P·V(j) has
    // completed; with two S buffers that wait is a step ahead of the softmax that needs it.
    // A descriptor's start-address field is bits 0-13 of (address >> 4); the tiles lie within
    // the first 256 KiB of shared memory, so a descriptor of (address + offset) is the
    // descriptor of the address plus (offset >> 4).
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tQ = tmem + kTmemQ;  // the tile's queries: column c holds dims 2c, 2c + 1
    // S(i) = Q K(i)ᵀ into the S buffer of step n0 + i; then the stage of K(i) is released
    auto issue_s = [&](int i) {
      const int e = ek(i);
      const uint32_t st = stage_of(e), b = (n0 + (uint32_t)i) & 1u;
      const uint64_t bd0 = sdesc_sw128(sRing + st * kSmemKTile, 16, kKGroupStride);
      const uint32_t dS = tmem + kTmemS + b * 128;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t boff = ((kk >> 2) * kKHalfOff + (kk & 3) * 32) >> 4;
        umma_ts(dS, tQ + kk * 8, bd0 + boff, kIdescS, kk > 0 ? 1u : 0u);
      }
      umma_commit(smem_u32(&ctl->s_full[b]));
      umma_commit(smem_u32(&ctl->kv_empty[st]));
    };
    // O (+)= P(j) V(j); then the stage of V(j) is released
    auto issue_pv = [&](int j) {
      const int e = ev(j);
      const uint32_t st = stage_of(e), b = (n0 + (uint32_t)j) & 1u;
      // V (block kk for keys 16kk..) is N-major: 64-column halves 2 KiB apart (LBO), 8-key
      // groups 1 KiB apart (SBO); P of keys 16kk.. is at column 8kk of the S buffer
      const uint64_t bd0 = sdesc_sw128(sRing + st * kSmemKTile, 2048, 1024);
      const uint32_t dS = tmem + kTmemS + b * 128, dO = tmem + kTmemO;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        umma_ts(dO, dS + kk * 8, bd0 + ((kk * kVBlockBytes) >> 4), kIdescPV,
                (j == 0 && kk == 0) ? 0u : 1u);
      umma_commit(smem_u32(&ctl->pv_done));
      umma_commit(smem_u32(&ctl->kv_empty[st]));
      if (j + 1 == ntiles) umma_commit(smem_u32(&ctl->o_done));
    };
    bool ok = mbar_wait(smem_u32(&ctl->q_full), ps.q_cnt & 1, wc);
    if (warp == 3) {
      // S(0), S(1), then S(j + 2) once P·V(j) has completed (completion n of pv_done: every one
      // is waited for, so the parity is unambiguous) and K(j + 2) has landed
      for (int i = 0; ok && i < 2 && i < ntiles; ++i) {
        ok = mbar_wait(smem_u32(&ctl->kv_full[stage_of(ek(i))]), phase_of(ek(i)), wc);
        tc_fence_after();
        if (ok && lane == 0) issue_s(i);
        __syncwarp();
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        const uint32_t n = n0 + j;
        ok = mbar_wait(smem_u32(&ctl->pv_done), n & 1, wc);
        if (!ok || j + 2 >= ntiles) continue;
        ok = mbar_wait(smem_u32(&ctl->kv_full[stage_of(ek(j + 2))]), phase_of(ek(j + 2)), wc);
        tc_fence_after();
        if (ok && lane == 0) issue_s(j + 2);
        __syncwarp();
      }
    } else {
      // P·V(j) once P(j) is written and V(j) has landed
      for (int j = 0; ok && j < ntiles; ++j) {
        const uint32_t n = n0 + j;
        ok = mbar_wait(smem_u32(&ctl->p_ready[n & 1]), (n >> 1) & 1, wc) &&
             mbar_wait(smem_u32(&ctl->kv_full[stage_of(ev(j))]), phase_of(ev(j)), wc);
        tc_fence_after();
        if (ok && lane == 0) issue_pv(j);
        __syncwarp();
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 8) {
    // ------------------------------------------------------------------ queries and softmax
    const int quarter = warp & 3;
    const int hf = (warp - kSoftmaxWarp0) >> 2;  // this thread's half of the keys and of O
    const int row = quarter * 32 + lane;         // the tile row (TMEM lane)
    const uint32_t trow = ctl->tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tO = trow + kTmemO + hf * (HD / 2);  // this half's O columns
    const uint32_t tX = trow + kTmemX;                  // the halves' exchange columns
    const int qi = t * p.tq + (row >> p.hp_log2);  // this row's token (in the chunk)
    const int h = h0 + (row & ((1 << p.hp_log2) - 1));      // and query head
    const bool valid = qi < qlen;
    const int lim = p.causal ? min(P + qi + 1, ke) : ke;  // keys [.., lim) are visible
    {
      // the row's queries (this half's dims; zeros past the chunk) into TMEM, bf16 pairs in the
      // order the S MMAs read them; one arrival per warp once its stores have completed
      constexpr int kWords = HD / 4;  // 32-bit words of half a row
      uint32_t qw[32];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q_prefill + ((size_t)(q0 + (valid ? qi : 0)) * p.Hq + h) * HD + hf * (HD / 2));
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = valid ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
      }
      if constexpr (HD == 128) tmem_st32(trow + kTmemQ + hf * kWords, qw);
      else tmem_st16(trow + kTmemQ + hf * kWords, qw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->q_full));
    }
    float m = -INFINITY, l = 0.f;  // the row's running max (log2 units), this half's sum
    bool ok = true;
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
    // scores of the half's 64 columns visible below v (others -inf)
    auto mask64 = [&](uint32_t(&a)[32], uint32_t(&b)[32], int v) {
      if (!__all_sync(0xffffffffu, v >= 64)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= v) a[c] = f2u(-INFINITY);
          if (c + 32 >= v) b[c] = f2u(-INFINITY);
        }
      }
    };
    auto max64 = [](const uint32_t(&a)[32], const uint32_t(&b)[32]) {
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmax3(u2f(a[i]), u2f(a[i + 8]), u2f(a[i + 16]));
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], u2f(a[i + 24]), u2f(b[i]));
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], u2f(b[i + 8]), u2f(b[i + 16]));
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], u2f(b[i + 24]));
      return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
    };
    // exponentials of the half's 64 scores against the reference max; P as bf16 pairs at
    // columns [pc, pc + 32) of the S buffer at tS; returns their sum
    auto exp64 = [&](const uint32_t(&a)[32], const uint32_t(&b)[32], float2 nm2, uint32_t tS,
                     uint32_t pc) {
      float2 sum[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sum[i] = make_float2(0.f, 0.f);
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float2 xv = ffma2(make_float2(u2f(a[2 * c]), u2f(a[2 * c + 1])), c2, nm2);
        const float2 e = make_float2(ex2(xv.x), ex2(xv.y));
        sum[c & 3] = fadd2(sum[c & 3], e);
        pk[c] = pack_bf16x2(e.x, e.y);
      }
      tmem_st16(tS + pc, pk);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float2 xv = ffma2(make_float2(u2f(b[2 * c]), u2f(b[2 * c + 1])), c2, nm2);
        const float2 e = make_float2(ex2(xv.x), ex2(xv.y));
        sum[c & 3] = fadd2(sum[c & 3], e);
        pk[c] = pack_bf16x2(e.x, e.y);
      }
      tmem_st16(tS + pc + 16, pk);
      const float2 s01 = fadd2(fadd2(sum[0], sum[1]), fadd2(sum[2], sum[3]));
      return s01.x + s01.y;
    };
    // The other half's value of this row through TMEM column `col` (this half writes
    // col + hf, reads col + 1 - hf); both halves of every row pass the same barrier.
    auto exchange = [&](uint32_t col, float mine) {
      tmem_st1(tX + col + hf, f2u(mine));
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(2, 256);
      tc_fence_after();
      const uint32_t o = tmem_ld1(tX + col + (hf ^ 1));
      tmem_ld_wait();
      return u2f(o);
    };
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t n = n0 + j, b = n & 1;
      // After a failed wait the loop still runs (every wait then fails at once), so that the
      // warps pass the same barriers whatever happened.
      ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&ctl->s_full[b]), (n >> 1) & 1, wc));
      tc_fence_after();
      const uint32_t tS = trow + kTmemS + b * 128;
      const int vis = lim - (kb + j * kTileN) - hf * 64;  // visible columns of the half: [0, vis)
      uint32_t sa[32], sb[32];
      tmem_ld32(tS + hf * 64, sa);
      tmem_ld32(tS + hf * 64 + 32, sb);
      tmem_ld_wait();
      mask64(sa, sb, vis);
      const float mine = max64(sa, sb);
      // the row's max over both halves (exchange columns alternate with the step's parity, so
      // a half never overwrites a value its partner has yet to read)
      const float mx = fmaxf(mine, exchange(2 * b, mine));
      // scale > 0, so the max of the scaled scores is the scaled max
      const float m_new = fmaxf(m, mx * p.scale_log2);
      const bool resc = m_new > m + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2(m - m_new);
        m = m_new;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // O holds P·V of the earlier steps once P·V(n - 1) has completed (completion n - 1 of
        // pv_done; S(n), which this step waited for, was issued after P·V(n - 2), so the
        // barrier is at completion n - 1 or n: its parity is unambiguous)
        ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&ctl->pv_done), (n - 1) & 1, wc));
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < HD / 64; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + ch * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st32(tO + ch * 32, o);
        }
        tmem_st_wait();
      }
      const float mref = m == -INFINITY ? 0.f : m;
      l = l * alpha + exp64(sa, sb, make_float2(-mref, -mref), tS, hf * 32);
      tmem_st_wait();
      // every lane's P stores have completed; one arrival per warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_ready[b]));
    }
    if (ok) {  // the last P·V (and with it every MMA of the item)
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done), ps.q_cnt & 1, wc));
      tc_fence_after();
    }
    // the row sum over both halves
    const float lrow = l + exchange(4, l);
    // ------------------------------------------------------------------ epilogue
    // Each thread writes its half of the row's O columns.
    if (unit < 0) {
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
      uint16_t* dst = p.o_prefill + ((size_t)(q0 + qi) * p.Hq + h) * HD + hf * (HD / 2);
#pragma unroll 1
      for (int ch = 0; ch < HD / 64; ++ch) {
        uint32_t a[32];
        tmem_ld32(tO + ch * 32, a);
        tmem_ld_wait();
        if (valid && ok) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(u2f(a[2 * i]) * inv, u2f(a[2 * i + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    } else {
      const int nsplit = p.units[unit * kUnitWords + 0];
      const int slot0 = p.units[unit * kUnitWords + 1];
      uint8_t* const slots = reinterpret_cast<uint8_t*>(p.partial_p);
      uint8_t* slot = slots + (size_t)(slot0 + split) * kPrefillSlotBytes;
      // The partial is O / l in bf16 (the final output's precision) with the row's m and l in
      // fp32, written with streaming stores so that it does not push K/V tiles out of L2. O is
      // stored in 8-column chunks interleaved across the 32 rows of a warp (chunk c of row r at
      // uint4 ((r / 32) * 16 + c) * 32 + r % 32), so that each store and each load of the merge
      // moves 512 contiguous bytes per warp. This half holds chunks [c0, c0 + HD / 16).
      const size_t row_off = (size_t)(row >> 5) * (kHeadDim / 8) * 32 + (row & 31);
      const int c0 = hf * (HD / 16);
      uint4* o8 = reinterpret_cast<uint4*>(slot) + row_off;
      const float inv_l = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll 1
      for (int ch = 0; ch < HD / 64 && ok; ++ch) {
        uint32_t a[32];
        tmem_ld32(tO + ch * 32, a);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 4; ++i)
          __stcs(o8 + (c0 + ch * 4 + i) * 32,
                 make_uint4(pack_bf16x2(u2f(a[8 * i]) * inv_l, u2f(a[8 * i + 1]) * inv_l),
                            pack_bf16x2(u2f(a[8 * i + 2]) * inv_l, u2f(a[8 * i + 3]) * inv_l),
                            pack_bf16x2(u2f(a[8 * i + 4]) * inv_l, u2f(a[8 * i + 5]) * inv_l),
                            pack_bf16x2(u2f(a[8 * i + 6]) * inv_l, u2f(a[8 * i + 7]) * inv_l)));
      }
      constexpr int kMlOff = kTileM * kHeadDim * 2;  // m[128] then l[128], fp32
      if (ok && hf == 0) {
        float* ml = reinterpret_cast<float*>(slot + kMlOff);
        __stcs(ml + row, m);
        __stcs(ml + kTileM + row, lrow);
      }
      __threadfence();
      named_bar_sync(2, 256);
      if (row == 0 && hf == 0)
        ctl->merge_last[0] = ok && (atomicAdd(&p.arrive[unit], 1) == nsplit - 1);
      named_bar_sync(2, 256);
      if (ctl->merge_last[0] && ok) {
        __threadfence();
        if (valid) {
          // the planner makes at most kMaxPrefillSplits splits; all loads of one pass are
          // independent, so each pass costs one memory latency rather than one per split.
          // Split k weighs 2^(m_k - m*) l_k (its O / l is stored).
          const uint8_t* base = slots + (size_t)slot0 * kPrefillSlotBytes;
          float f[kMaxPrefillSplits];
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < kMaxPrefillSplits; ++k) {
            f[k] = k < nsplit
                       ? __ldcg(reinterpret_cast<const float*>(base + (size_t)k * kPrefillSlotBytes + kMlOff) + row)
                       : -INFINITY;
            mx = fmaxf(mx, f[k]);
          }
          float den = 0.f;
#pragma unroll
          for (int k = 0; k < kMaxPrefillSplits; ++k) {
            const float lk =
                k < nsplit ? __ldcg(reinterpret_cast<const float*>(base + (size_t)k * kPrefillSlotBytes + kMlOff) +
                                    kTileM + row)
                           : 0.f;
            f[k] = f[k] == -INFINITY ? 0.f : ex2(f[k] - mx) * lk;  // weight of split k
            den += f[k];
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          uint16_t* dst = p.o_prefill + ((size_t)(q0 + qi) * p.Hq + h) * HD;
#pragma unroll 1
          for (int ch = hf * (HD / 32); ch < (hf + 1) * (HD / 32); ++ch) {  // 16 columns at a time
            float acc[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxPrefillSplits; ++k) {
              if (k < nsplit) {
                const uint4* src = reinterpret_cast<const uint4*>(base + (size_t)k * kPrefillSlotBytes) +
                                   row_off + (size_t)ch * 2 * 32;
                const float fk = f[k] * inv;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                  const uint4 v = __ldcs(src + c * 32);
#pragma unroll
                  for (int w = 0; w < 4; ++w) {
                    const uint32_t u = u4_word(v, w);
                    acc[8 * c + 2 * w] += fk * bf16lo(u);
                    acc[8 * c + 2 * w + 1] += fk * bf16hi(u);
                  }
                }
              }
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 16);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              d4[i] = make_uint4(pack_bf16x2(acc[8 * i], acc[8 * i + 1]),
                                 pack_bf16x2(acc[8 * i + 2], acc[8 * i + 3]),
                                 pack_bf16x2(acc[8 * i + 4], acc[8 * i + 5]),
                                 pack_bf16x2(acc[8 * i + 6], acc[8 * i + 7]));
          }
        }
        if (row == 0 && hf == 0) p.arrive[unit] = 0;  // ready for the next run
      }
    }
    tc_fence_before();
  }
  // every thread of the prefill slot keeps the same pipeline positions
  ps.q_cnt++;
  ps.t_cnt += ntiles;
  named_bar_sync(1, kPrefillThreads);
}

// ============================================================================ decode item
// Reduce-scatter of 16 per-row partial dot products over the 32 lanes of a warp (each lane
// holds 4 of the 128 dims): five butterfly steps halve the values per lane, the last one adds
// the lane pair. Afterwards lanes 2r and 2r+1 both hold the full dot product of row r.
__device__ __forceinline__ float rowdot_scatter(float (&v)[16], int lane) {
  float a[8];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = hi ? v[i] : v[i + 8];
      const float keep = hi ? v[i + 8] : v[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  float b[4];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = hi ? a[i] : a[i + 4];
      const float keep = hi ? a[i + 4] : a[i];
      b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  float c[2];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = hi ? b[i] : b[i + 2];
      const float keep = hi ? b[i + 2] : b[i];
      c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  const bool hi = lane & 2;
  const float send = hi ? c[0] : c[1];
  const float keep = hi ? c[1] : c[0];
  float d = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

constexpr int kScr = kHeadDim + 4;  // shared scratch row of one warp and head: o[128], m, l
constexpr int kRow = kHeadDim + 2;  // global partial slot row: o[128], m, l

// DL consecutive bf16 values of one lane (DL = head dim / 32: 4 or 2), as one vector load.
template <int DL> struct LaneVec;
template <> struct LaneVec<4> {
  uint2 v;
  __device__ __forceinline__ void load(const uint16_t* src) { v = *reinterpret_cast<const uint2*>(src); }
  __device__ __forceinline__ float operator[](int i) const {
    return i == 0 ? bf16lo(v.x) : i == 1 ? bf16hi(v.x) : i == 2 ? bf16lo(v.y) : bf16hi(v.y);
  }
  __device__ __forceinline__ void zero() { v = make_uint2(0, 0); }
};
template <> struct LaneVec<2> {
  uint32_t v;
  __device__ __forceinline__ void load(const uint16_t* src) { v = *reinterpret_cast<const uint32_t*>(src); }
  __device__ __forceinline__ float operator[](int i) const { return i == 0 ? bf16lo(v) : bf16hi(v); }
  __device__ __forceinline__ void zero() { v = 0; }
};

// Decode, MHA (one query head per kv-head): CUDA-core path. Each warp streams its blocks with
// bulk copies of whole (block, kv-head) units; q lives in registers (HD/32 dims per lane); q·k is
// reduce-scattered across the warp with shuffles. Leaves the warp's (o, m, l) in the shared
// scratch; returns false on abort.
// Block-table entries of one decode warp's blocks (block i of the warp is entry i * nw of
// `row`), read 32 at a time, one window ahead: lane j holds the entry of block 32 w + j, so the
// copy of a block never waits on a global load of its entry. at(i) must be called by all 32
// lanes with i = 0, 1, 2, ... in order.
struct BtWindow {
  const int32_t* row;
  int nw, n;
  int cur = 0, nxt = 0;
  __device__ int load(int first, int lane) const {
    const int j = first + lane;
    return j < n ? __ldg(row + (size_t)j * nw) : 0;
  }
  __device__ void init(int lane) {
    cur = load(0, lane);
    nxt = load(32, lane);
  }
  __device__ int at(int i, int lane) {
    if (i >= 32 && (i & 31) == 0) {
      cur = nxt;
      nxt = load(i + 32, lane);
    }
    return __shfl_sync(0xffffffffu, cur, i & 31);
  }
};

template <int GT, int HD>
__device__ bool decode_simt(const Params& p, const int32_t* it, const DecodeCtx& dc,
                            SmemCtl* ctl, PipeState& ps, const WaitCtx& wc) {
  constexpr int DL = HD / 32;                    // dims per lane
  constexpr uint32_t kUnit = kBlockSize * HD * 2;  // bytes of one (block, kv-head) K or V unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = warp - dc.w0;  // this warp's index among the item's warps
  const int d = it[1], g = it[2], kb = it[4], ke = it[5];
  const int G = p.G;
  const int32_t* bt_row = p.block_tables + (size_t)(p.Np + d) * p.maxb;
  const int nblk = (ke - kb + kBlockSize - 1) / kBlockSize;
  const int blk0 = kb / kBlockSize;
  const bool mine = wl >= 0 && wl < dc.nw;
  int nmine = mine && nblk > wl ? (nblk - wl + dc.nw - 1) / dc.nw : 0;
  {  // the sequence's last row (this step's token) may be appended by this launch
    int oka = 1;
    if (lane == 0 && nmine > 0 && ke >= p.kv_lens[p.Np + d]) oka = wait_appended(p, ps, wc);
    if (!__shfl_sync(0xffffffffu, oka, 0)) nmine = 0;
  }
  uint8_t* ring = dc.ring + (mine ? wl : 0) * kDecodeSlots * kSmemDecodeSlot;
  float* ps_x = dc.scores + (mine ? wl : 0) * kMaxGroup * kBlockSize;

  // q in registers: DL consecutive dims per lane, premultiplied by scale*log2(e)
  float q[GT][DL], o[GT][DL], m[GT], ls[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m[h] = -INFINITY;
    ls[h] = 0.f;
#pragma unroll
    for (int k = 0; k < DL; ++k) o[h][k] = q[h][k] = 0.f;
    if (h < G) {
      LaneVec<DL> r;
      r.load(p.q_decode + ((size_t)d * p.Hq + (size_t)g * G + h) * HD + lane * DL);
#pragma unroll
      for (int k = 0; k < DL; ++k) q[h][k] = r[k] * p.scale_log2;
    }
  }

  const uint64_t pol = policy_evict_first();
  BtWindow bt{bt_row + blk0 + wl, dc.nw, nmine};
  bt.init(lane);
  auto issue = [&](int i, int phys) {  // lane 0 only: block i of this warp into slot i % 2
    const int slot = i & 1;
    if (phys < 0 || phys >= p.num_blocks) {
      record_error(p.status, POD_ATTN_ERR_BAD_INDEX);
      phys = 0;
    }
    const size_t off = ((size_t)phys * p.Hkv + g) * (kBlockSize * HD);
    const uint32_t bar = smem_u32(&ctl->dslot[warp][slot]);
    const uint32_t dst = smem_u32(ring + slot * kSmemDecodeSlot);
    mbar_arrive_expect_tx(bar, 2 * kUnit);
    bulk_load(dst, p.k_pool + off, kUnit, bar, pol);
    bulk_load(dst + kSmemDecodeSlot / 2, p.v_pool + off, kUnit, bar, pol);
  };
  {
    const int ph0 = bt.at(0, lane), ph1 = bt.at(1, lane);
    if (lane == 0) {
      if (nmine > 0) issue(0, ph0);
      if (nmine > 1) issue(1, ph1);
    }
  }
  bool ok = true;
  const int r = lane >> 1;  // the row whose full score this lane holds after the reduction
  for (int i = 0; i < nmine; ++i) {
    const int slot = i & 1;
    // every lane takes the same exit, so the warp's shuffles below stay converged
    const bool got = mbar_wait(smem_u32(&ctl->dslot[warp][slot]), (ps.dphase >> slot) & 1, wc,
                               kSleepNs);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    ps.dphase ^= 1u << slot;
    const int key0 = kb + (wl + i * dc.nw) * kBlockSize;
    const int nv = min(kBlockSize, ke - key0);
    const uint16_t* Ks = reinterpret_cast<const uint16_t*>(ring + slot * kSmemDecodeSlot);
    const uint16_t* Vs = Ks + kBlockSize * kHeadDim;
    LaneVec<DL> kr[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) kr[c].load(Ks + c * HD + lane * DL);
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      if (h < G) {
        float part[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          part[c] = 0.f;
#pragma unroll
          for (int k = 0; k < DL; ++k) part[c] += q[h][k] * kr[c][k];
        }
        float sc = rowdot_scatter(part, lane);
        sc = r < nv ? sc : -INFINITY;
        float bm = sc;
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        if (bm > m[h]) {  // warp-uniform
          const float alpha = ex2(m[h] - bm);
          m[h] = bm;
          ls[h] *= alpha;
#pragma unroll
          for (int k = 0; k < DL; ++k) o[h][k] *= alpha;
        }
        const float pv = r < nv ? ex2(sc - m[h]) : 0.f;
        if ((lane & 1) == 0) {
          ls[h] += pv;
          ps_x[h * kBlockSize + r] = pv;
        }
      }
    }
    __syncwarp();
    LaneVec<DL> vr[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) vr[c].load(Vs + c * HD + lane * DL);
    if (nv < kBlockSize) {
      // rows past the sequence end may hold anything; their weight is 0 and so is their value
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c >= nv) vr[c].zero();
    }
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      if (h < G) {
        const float4* pp = reinterpret_cast<const float4*>(ps_x + h * kBlockSize);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const float4 w = pp[c4];
          const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int k = 0; k < DL; ++k) o[h][k] += wv[e] * vr[c4 * 4 + e][k];
        }
      }
    }
    __syncwarp();
    {
      const int ph = bt.at(i + 2, lane);
      if (lane == 0 && i + 2 < nmine) issue(i + 2, ph);
    }
  }
#pragma unroll
  for (int h = 0; h < GT; ++h) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) ls[h] += __shfl_xor_sync(0xffffffffu, ls[h], off);
  }

  // ---- leave the warp's partial state (ring memory is free once every warp is done) ----
  named_bar_sync(dc.bar_id, dc.bar_threads);
  float* scr = reinterpret_cast<float*>(dc.ring);  // [nw][GT][kScr]
  if (ok && mine) {
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      if (h < G) {
        float* dst = scr + (wl * GT + h) * kScr;
#pragma unroll
        for (int k = 0; k < DL; ++k) dst[lane * DL + k] = o[h][k];
        if (lane == 0) {
          dst[kHeadDim] = m[h];
          dst[kHeadDim + 1] = ls[h];
        }
      }
    }
  }
  return ok;
}

// Decode, grouped-query attention (G >= 2 query heads per kv-head): warp-level tensor-core MMAs
// (m16n8k16, bf16 in, fp32 accumulate). Each warp streams its blocks through TMA (one 16-row x
// 64-dim box per half, 128-byte swizzle, so ldmatrix reads are free of bank conflicts); per
// 16-key block: S = Q·Kᵀ with the G heads as rows (2 x 8 MMAs), a row softmax over 16 keys with
// quad shuffles, then Oᵀ += Vᵀ·Pᵀ (8 MMAs) with the heads as columns, so P goes from the S
// accumulators straight into the B operand and the accumulator needs only 32 registers.
template <int GT, int HD>
__device__ bool decode_tc(const Params& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                          const int32_t* it, const DecodeCtx& dc, SmemCtl* ctl, PipeState& ps,
                          const WaitCtx& wc) {
  constexpr int kKS = HD / 16;     // k-steps of S = Q Kᵀ and 16-dim tiles of Oᵀ
  constexpr int kHalves = HD / 64; // 64-dim halves of a K or V block in the slot
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = warp - dc.w0;  // this warp's index among the item's warps
  const int d = it[1], g = it[2], kb = it[4], ke = it[5];
  const int G = p.G;
  const int32_t* bt_row = p.block_tables + (size_t)(p.Np + d) * p.maxb;
  const int nblk = (ke - kb + kBlockSize - 1) / kBlockSize;
  const int blk0 = kb / kBlockSize;
  const bool mine = wl >= 0 && wl < dc.nw;
  int nmine = mine && nblk > wl ? (nblk - wl + dc.nw - 1) / dc.nw : 0;
  {  // the sequence's last row (this step's token) may be appended by this launch
    int oka = 1;
    if (lane == 0 && nmine > 0 && ke >= p.kv_lens[p.Np + d]) oka = wait_appended(p, ps, wc);
    if (!__shfl_sync(0xffffffffu, oka, 0)) nmine = 0;
  }
  uint8_t* ring = dc.ring + (mine ? wl : 0) * kDecodeSlots * kSmemDecodeSlot;
  const uint32_t ring_s = smem_u32(ring);
  const int hr = lane >> 2, qd = lane & 3;  // fragment row (query head) and quad lane

  // A fragments of Q: row hr = head g*G + hr (rows >= G and rows 8..15 are zero)
  uint32_t qa0[kKS], qa2[kKS];
#pragma unroll
  for (int ks = 0; ks < kKS; ++ks) qa0[ks] = qa2[ks] = 0u;
  if (hr < G) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(
        p.q_decode + ((size_t)d * p.Hq + (size_t)g * G + hr) * HD);
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      qa0[ks] = qw[ks * 8 + qd];
      qa2[ks] = qw[ks * 8 + qd + 4];
    }
  }
  float ot[kKS][4];  // Oᵀ: dims 16mt + hr (+8) x heads 2qd, 2qd+1
#pragma unroll
  for (int mt = 0; mt < kKS; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
  float m = -INFINITY, l = 0.f;

  BtWindow bt{bt_row + blk0 + wl, dc.nw, nmine};
  bt.init(lane);
  const uint64_t pol = policy_evict_first();  // decode K/V is read once: keep L2 for the rest
  auto issue = [&](int i, int phys) {  // lane 0 only: block i of this warp into slot i % 2
    const int slot = i & 1;
    if (phys < 0 || phys >= p.num_blocks) {
      record_error(p.status, POD_ATTN_ERR_BAD_INDEX);
      phys = 0;
    }
    const int y = (phys * p.Hkv + g) * kBlockSize;
    const uint32_t bar = smem_u32(&ctl->dslot[warp][slot]);
    const uint32_t dst = ring_s + slot * kSmemDecodeSlot;
    mbar_arrive_expect_tx(bar, 2 * kBlockSize * HD * 2);
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) {  // K at +0, V at +4 KiB; 64-dim halves 2 KiB apart
      tma_load_2d_hint(dst + hf * 2048, tmk, bar, 64 * hf, y, pol);
      tma_load_2d_hint(dst + 4096 + hf * 2048, tmv, bar, 64 * hf, y, pol);
    }
  };
  {
    const int ph0 = bt.at(0, lane), ph1 = bt.at(1, lane);
    if (lane == 0) {
      if (nmine > 0) issue(0, ph0);
      if (nmine > 1) issue(1, ph1);
    }
  }
  bool ok = true;
  const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
  for (int i = 0; i < nmine; ++i) {
    const int slot = i & 1;
    // every lane takes the same exit, so the warp's shuffles below stay converged
    const bool got = mbar_wait(smem_u32(&ctl->dslot[warp][slot]), (ps.dphase >> slot) & 1, wc,
                               kSleepNs);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    ps.dphase ^= 1u << slot;
    const int key0 = kb + (wl + i * dc.nw) * kBlockSize;
    const int nv = min(kBlockSize, ke - key0);
    const uint32_t Ks = ring_s + slot * kSmemDecodeSlot, Vs = Ks + 4096;
    if (nv < kBlockSize) {
      // rows past the sequence end may hold anything (even NaN): zero those V rows, since
      // their weight 0 times NaN would not be 0
      uint8_t* vb = ring + slot * kSmemDecodeSlot + 4096;
      for (int c = lane; c < (kBlockSize - nv) * 8 * kHalves; c += 32) {
        const int r = nv + c / (8 * kHalves), half = (c >> 3) % kHalves, ch = c & 7;
        *reinterpret_cast<uint4*>(vb + half * 2048 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    // S = Q Kᵀ: keys 0-7 in s0, keys 8-15 in s1
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const int key = (mi >> 1) * 8 + mr, ch = (ks & 3) * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(Ks + (ks >> 2) * 2048 + key * 128 + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
      const uint32_t a[4] = {qa0[ks], 0u, qa2[ks], 0u};
      mma_16816(s0, a, b0, b1);
      mma_16816(s1, a, b2, b3);
    }
    // this lane's scores: keys 2qd, 2qd+1, 8+2qd, 9+2qd of row hr
    float x[4] = {s0[0], s0[1], s1[0], s1[1]};
    const int kx[4] = {2 * qd, 2 * qd + 1, 8 + 2 * qd, 9 + 2 * qd};
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = kx[e] < nv ? x[e] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, x[e]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const bool resc = m_new > m + 8.f;  // lazy rescale, as in the prefill tiles
    float alpha = 1.f;
    if (resc) {
      alpha = ex2(m - m_new);
      m = m_new;
    }
    if (__any_sync(0xffffffffu, resc)) {
      l *= alpha;
      // Oᵀ columns are heads 2qd and 2qd+1: their factors live in rows (lanes) 8qd and 8qd+4
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * qd);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * qd + 4);
#pragma unroll
      for (int mt = 0; mt < kKS; ++mt) {
        ot[mt][0] *= a0;
        ot[mt][1] *= a1;
        ot[mt][2] *= a0;
        ot[mt][3] *= a1;
      }
    }
    const float mref = m == -INFINITY ? 0.f : m;
    float pr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pr[e] = ex2(x[e] - mref);
      l += pr[e];
    }
    // Pᵀ as the B operand (keys x heads): exactly this lane's S values, packed
    const uint32_t pb0 = pack_bf16x2(pr[0], pr[1]), pb1 = pack_bf16x2(pr[2], pr[3]);
    // Oᵀ += Vᵀ Pᵀ: A = Vᵀ tiles of 16 dims x 16 keys, ldmatrix-transposed from the V slot
#pragma unroll
    for (int mt = 0; mt < kKS; ++mt) {
      const int key = (mi >> 1) * 8 + mr, ch = (mt & 3) * 2 + (mi & 1);
      uint32_t a[4];
      ldsm_x4_t(Vs + (mt >> 2) * 2048 + key * 128 + ((ch ^ (key & 7)) << 4), a[0], a[1], a[2],
                a[3]);
      mma_16816(ot[mt], a, pb0, pb1);
    }
    __syncwarp();
    {
      const int ph = bt.at(i + 2, lane);
      if (lane == 0 && i + 2 < nmine) issue(i + 2, ph);
    }
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);

  named_bar_sync(dc.bar_id, dc.bar_threads);
  float* scr = reinterpret_cast<float*>(dc.ring);  // [nw][GT][kScr]
  if (ok && mine) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int head = 2 * qd + e;
      if (head < G) {
        float* dst = scr + (wl * GT + head) * kScr;
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) {
          dst[mt * 16 + hr] = ot[mt][e];
          dst[mt * 16 + hr + 8] = ot[mt][2 + e];
        }
      }
    }
    if (hr < G && qd == 0) {
      float* dst = scr + (wl * GT + hr) * kScr;
      dst[kHeadDim] = m;
      dst[kHeadDim + 1] = l;
    }
  }
  return ok;
}

// ---------------------------------------------------------------- FP8 cache decode
// Decode over an e4m3 cache with per-channel K and per-token V scales ("LLMSO - W4 -
// Optimization & Frameworks", §"2-4. 고급 KV 캐싱 기법"), head dim 128, on the warp tensor
// cores in f16: every e4m3 value is
// an f16 value, so one conversion per pair of values feeds the MMA exactly. The per-channel K
// scale is folded into q once per item (q' = q * k_scale), the per-token V scale into the P·V
// weights (the row sum keeps the unscaled weights).
//
// Each warp streams whole (block, kv-head) units: the K and V tiles (16 rows x 128 bytes each) by
// TMA with the 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r & 7)) and the 16 V
// scales by bulk copy, into a ring of 3 slots (MHA) or 2 (GQA). The lanes read their MMA
// operands straight from the tiles, in a channel order of their own that makes each read a
// contiguous 16-byte chunk and the reads of a quarter-warp fall in distinct banks:
//  * S = q' Kᵀ: in k-step ks, lane (g = lane / 4, t = lane % 4) holds channels 32t + 4ks .. +3
//    of its key row(s) g (and g + 8) as the B fragment, and q' is permuted to match;
//  * Oᵀ += Vᵀ Pᵀ: lane (g, t) holds channels 16g .. 16g + 15 of its four keys 2t, 2t+1, 2t+8,
//    2t+9; output row g (g + 8) of m-tile mt is channel 16g + 2mt (+ 1).
constexpr int kFp8Tile = kBlockSize * 128;                          // 2 KiB: one K or V tile
constexpr int kFp8Slot = 2 * kFp8Tile;                              // K then V (1 KiB-aligned)
constexpr int kFp8Ring = kDecodeSlotsFp8 * kFp8Slot;                // 12 KiB per warp
constexpr int kFp8ScaleBytes = kDecodeSlotsFp8 * kBlockSize * 4;    // V scales of the slots
constexpr int kFp8GroupBytes = 49 * 1024;  // 4 rings + 4 scale areas, rounded to 1 KiB
constexpr int kFp8Groups = 4;              // warps 0-3, 4-7, 8-11 and the decode slot 12-15
static_assert(kDecodeWarps * (kFp8Ring + kFp8ScaleBytes) <= kFp8GroupBytes, "FP8 group size");
static_assert(2 * kMaxGroup * kMaxDecodeSplits + kMaxGroup <= kDecodeWarps * kFp8Ring / 4 &&
                  2 * kMaxGroup * kMaxDecodeSplits + kMaxGroup <= kSmemDecodeRing / 4,
              "the split merge's weights must fit a decode group's ring");
static_assert(kDecodeWarps * kMaxGroup * kScr * 4 <= kDecodeWarps * kFp8Ring,
              "the combine scratch must fit the rings");
static_assert(kFp8Groups * kFp8GroupBytes + kFp8Groups * kDecodeWarps * kSmemScoresPerWarp <=
                  kSmemCtlOff,
              "four FP8 decode groups must fit below the control block");

template <int GT>
__device__ bool decode_tc_fp8(const Params& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                              const int32_t* it, const DecodeCtx& dc, SmemCtl* ctl, PipeState& ps,
                              const WaitCtx& wc) {
  constexpr int kKS = 8;
  // ring slots in use: three for MHA (one head per block: the least work per byte), two for GQA,
  // where a third measured slower (more copies in flight than the memory system serves better)
  constexpr int kSlots = GT == 1 ? kDecodeSlotsFp8 : 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wl = warp - dc.w0;
  const int d = it[1], g = it[2], kb = it[4], ke = it[5];
  const int G = p.G;
  const int32_t* bt_row = p.block_tables + (size_t)(p.Np + d) * p.maxb;
  const int nblk = (ke - kb + kBlockSize - 1) / kBlockSize;
  const int blk0 = kb / kBlockSize;
  const bool mine = wl >= 0 && wl < dc.nw;
  const int nmine = mine && nblk > wl ? (nblk - wl + dc.nw - 1) / dc.nw : 0;
  uint8_t* ring = dc.ring + (mine ? wl : 0) * kFp8Ring;
  const float* vscales =
      reinterpret_cast<const float*>(dc.ring + kDecodeWarps * kFp8Ring + (mine ? wl : 0) * kFp8ScaleBytes);
  const uint32_t ring_s = smem_u32(ring);
  const int hr = lane >> 2, qd = lane & 3;

  // A fragments of q' = q * k_scale, channels 32qd + 4ks + {0,1} (a0) and {2,3} (a2)
  uint32_t qa0[kKS], qa2[kKS];
#pragma unroll
  for (int ks = 0; ks < kKS; ++ks) qa0[ks] = qa2[ks] = 0u;
  if (hr < G) {
    const uint4* qv = reinterpret_cast<const uint4*>(
        p.q_decode + ((size_t)d * p.Hq + (size_t)g * G + hr) * 128 + 32 * qd);
    const float4* kv = reinterpret_cast<const float4*>(p.k_scale + (size_t)g * 128 + 32 * qd);
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // 8 channels per uint4: k-steps 2j and 2j + 1
      const uint4 w = qv[j];
      const float4 s0 = kv[2 * j], s1 = kv[2 * j + 1];
      qa0[2 * j] = pack_f16x2_sat(bf16lo(w.x) * s0.x, bf16hi(w.x) * s0.y);
      qa2[2 * j] = pack_f16x2_sat(bf16lo(w.y) * s0.z, bf16hi(w.y) * s0.w);
      qa0[2 * j + 1] = pack_f16x2_sat(bf16lo(w.z) * s1.x, bf16hi(w.z) * s1.y);
      qa2[2 * j + 1] = pack_f16x2_sat(bf16lo(w.w) * s1.z, bf16hi(w.w) * s1.w);
    }
  }
  float ot[kKS][4];  // Oᵀ: channels 16hr + 2mt (+1) x heads 2qd, 2qd+1
#pragma unroll
  for (int mt = 0; mt < kKS; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
  float m = -INFINITY, l = 0.f;

  BtWindow bt{bt_row + blk0 + wl, dc.nw, nmine};
  bt.init(lane);
  const uint64_t pol = policy_evict_first();  // the cache is read once: keep L2 for the rest
  auto issue = [&](int i, int phys) {  // lane 0 only: block i of this warp into slot i % kSlots
    const int slot = i % kSlots;
    if (phys < 0 || phys >= p.num_blocks) {
      record_error(p.status, POD_ATTN_ERR_BAD_INDEX);
      phys = 0;
    }
    const size_t unit = (size_t)phys * p.Hkv + g;
    const uint32_t bar = smem_u32(&ctl->dslot[warp][slot]);
    const uint32_t dst = ring_s + slot * kFp8Slot;
    mbar_arrive_expect_tx(bar, kFp8Slot + kBlockSize * 4);
    tma_load_2d_hint(dst, tmk, bar, 0, (int)(unit * kBlockSize), pol);
    tma_load_2d_hint(dst + kFp8Tile, tmv, bar, 0, (int)(unit * kBlockSize), pol);
    bulk_load(smem_u32(vscales + slot * kBlockSize), p.v_scale + unit * kBlockSize,
              kBlockSize * 4, bar, pol);
  };
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    const int ph = bt.at(i, lane);
    if (lane == 0 && nmine > i) issue(i, ph);
  }
  bool ok = true;
  const int kx[4] = {2 * qd, 2 * qd + 1, 8 + 2 * qd, 9 + 2 * qd};  // this lane's keys (S, P, V)
  for (int i = 0, slot = 0; i < nmine; ++i, slot = slot == kSlots - 1 ? 0 : slot + 1) {
    // every lane takes the same exit, so the warp's shuffles below stay converged
    const bool got = mbar_wait(smem_u32(&ctl->dslot[warp][slot]), (ps.dphase >> slot) & 1, wc,
                               kSleepNs);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    ps.dphase ^= 1u << slot;
    const int key0 = kb + (wl + i * dc.nw) * kBlockSize;
    const int nv = min(kBlockSize, ke - key0);
    const uint8_t* Kt = ring + slot * kFp8Slot;
    const uint8_t* Vt = Kt + kFp8Tile;
    // K rows hr and hr + 8: chunks 2qd, 2qd + 1 (swizzled by the row, whose low bits are hr)
    uint4 kw[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        kw[j][h] = *reinterpret_cast<const uint4*>(Kt + (hr + 8 * j) * 128 + (((2 * qd + h) ^ hr) << 4));
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const uint32_t w0 = u4_word(kw[0][ks >> 2], ks & 3), w1 = u4_word(kw[1][ks >> 2], ks & 3);
      const uint32_t a[4] = {qa0[ks], 0u, qa2[ks], 0u};
      mma_16816_f16(s0, a, e4m3x2_to_f16x2(w0 & 0xFFFFu), e4m3x2_to_f16x2(w0 >> 16));
      mma_16816_f16(s1, a, e4m3x2_to_f16x2(w1 & 0xFFFFu), e4m3x2_to_f16x2(w1 >> 16));
    }
    float x[4] = {s0[0], s0[1], s1[0], s1[1]};
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = kx[e] < nv ? x[e] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, x[e]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const bool resc = m_new > m + 8.f;
    float alpha = 1.f;
    if (resc) {
      alpha = ex2(m - m_new);
      m = m_new;
    }
    if (__any_sync(0xffffffffu, resc)) {
      l *= alpha;
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * qd);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * qd + 4);
#pragma unroll
      for (int mt = 0; mt < kKS; ++mt) {
        ot[mt][0] *= a0;
        ot[mt][1] *= a1;
        ot[mt][2] *= a0;
        ot[mt][3] *= a1;
      }
    }
    // V rows kx[0..3]: chunk hr (read after S, so the K and V words are never live together)
    uint4 vw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      vw[k] = *reinterpret_cast<const uint4*>(Vt + kx[k] * 128 + ((hr ^ (kx[k] & 7)) << 4));
    float vsc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) vsc[k] = vscales[slot * kBlockSize + kx[k]];
    __syncwarp();
    // the slot is read: refill it with the block kSlots ahead
    {
      const int ph = bt.at(i + kSlots, lane);
      if (lane == 0 && i + kSlots < nmine) issue(i + kSlots, ph);
    }
    if (nv < kBlockSize) {  // rows past the end may hold anything (even NaN): weight-0 V is 0
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (kx[k] >= nv) vw[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    const float mref = m == -INFINITY ? 0.f : m;
    float pw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pr = ex2(x[e] - mref);
      l += pr;
      pw[e] = kx[e] < nv ? fminf(pr * vsc[e], kF16Max) : 0.f;  // P·V weight: P x V scale
    }
    const uint32_t pb0 = pack_f16x2(pw[0], pw[1]);
    const uint32_t pb1 = pack_f16x2(pw[2], pw[3]);
#pragma unroll
    for (int mt = 0; mt < kKS; ++mt) {
      // channels 16hr + 2mt, +1 of keys (kx0, kx1) and (kx2, kx3): bytes 2(mt&1), 2(mt&1)+1
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
      const uint32_t u01 = __byte_perm(u4_word(vw[0], mt >> 1), u4_word(vw[1], mt >> 1), sel);
      const uint32_t u23 = __byte_perm(u4_word(vw[2], mt >> 1), u4_word(vw[3], mt >> 1), sel);
      const uint32_t a[4] = {e4m3x2_to_f16x2(u01 & 0xFFFFu), e4m3x2_to_f16x2(u01 >> 16),
                             e4m3x2_to_f16x2(u23 & 0xFFFFu), e4m3x2_to_f16x2(u23 >> 16)};
      mma_16816_f16(ot[mt], a, pb0, pb1);
    }
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  named_bar_sync(dc.bar_id, dc.bar_threads);
  float* scr = reinterpret_cast<float*>(dc.ring);  // [nw][GT][kScr]
  if (ok && mine) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int head = 2 * qd + e;
      if (head < G) {
        float* dst = scr + (wl * GT + head) * kScr + 16 * hr;
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt)
          *reinterpret_cast<float2*>(dst + 2 * mt) = make_float2(ot[mt][e], ot[mt][2 + e]);
      }
    }
    if (hr < G && qd == 0) {
      float* dst = scr + (wl * GT + hr) * kScr;
      dst[kHeadDim] = m;
      dst[kHeadDim + 1] = l;
    }
  }
  return ok;
}

// Append of one new token per decode sequence to an e4m3 cache. One warp per (sequence,
// kv-head), 4 channels per lane. K: e4m3(k / k_scale[g][c]); V: scale = max |v| / 448 over the
// row (1 if 0), e4m3(v / scale). Divisions are IEEE binary32 (round to nearest), so the codes
// are decided in the precision the format's reference quantiser uses.
struct AppendFp8Args {
  const uint16_t* k_new;  // bf16 [Nd][Hkv][128]
  const uint16_t* v_new;
  uint8_t* k8;            // e4m3 [NB][Hkv][16][128]
  uint8_t* v8;
  const float* k_scale;   // [Hkv][128]
  float* v_scale;         // [NB][Hkv][16]
  const int32_t* block_tables;
  const int32_t* new_rows;  // (sequence, position) per new token
  int32_t* status;
  int n_new, Hkv, maxb, num_blocks;
};

__global__ void __launch_bounds__(256) append_fp8_kernel(const __grid_constant__ AppendFp8Args a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.n_new * a.Hkv;
  for (int u = blockIdx.x * 8 + warp; u < units; u += gridDim.x * 8) {
    const int tok = u / a.Hkv, g = u % a.Hkv;
    const int seq = a.new_rows[2 * tok], pos = a.new_rows[2 * tok + 1];
    const int phys = a.block_tables[(size_t)seq * a.maxb + pos / kBlockSize];
    if (phys < 0 || phys >= a.num_blocks) {
      if (lane == 0) record_error(a.status, POD_ATTN_ERR_BAD_INDEX);
      continue;
    }
    const size_t row = ((size_t)phys * a.Hkv + g) * kBlockSize + pos % kBlockSize;
    const size_t src = ((size_t)tok * a.Hkv + g) * 128 + lane * 4;
    const uint2 kw = *reinterpret_cast<const uint2*>(a.k_new + src);
    const uint2 vw = *reinterpret_cast<const uint2*>(a.v_new + src);
    const float4 ks = *reinterpret_cast<const float4*>(a.k_scale + (size_t)g * 128 + lane * 4);
    const float k[4] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y)};
    const float v[4] = {bf16lo(vw.x), bf16hi(vw.x), bf16lo(vw.y), bf16hi(vw.y)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float vs = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const uint32_t kq = (uint32_t)e4m3x2_from_f32(__fdiv_rn(k[0], ks.x), __fdiv_rn(k[1], ks.y)) |
                        ((uint32_t)e4m3x2_from_f32(__fdiv_rn(k[2], ks.z), __fdiv_rn(k[3], ks.w)) << 16);
    const uint32_t vq = (uint32_t)e4m3x2_from_f32(__fdiv_rn(v[0], vs), __fdiv_rn(v[1], vs)) |
                        ((uint32_t)e4m3x2_from_f32(__fdiv_rn(v[2], vs), __fdiv_rn(v[3], vs)) << 16);
    *reinterpret_cast<uint32_t*>(a.k8 + row * 128 + lane * 4) = kq;
    *reinterpret_cast<uint32_t*>(a.v8 + row * 128 + lane * 4) = vq;
    if (lane == 0) a.v_scale[row] = vs;
  }
}

// Combine the warps' states of a decode item, then write the output or the split's partial and,
// for the last split of a unit to arrive, merge all partials.
template <int GT, int HD, bool FP8>
__device__ void decode_item(const Params& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                            const int32_t* it, const DecodeCtx& dc, SmemCtl* ctl,
                            PipeState& ps, const WaitCtx& wc) {
  const int d = it[1], g = it[2], unit = it[6], split = it[7];
  const int G = p.G;
  const int ltid = threadIdx.x - dc.first_thread;
  if constexpr (FP8) {
    decode_tc_fp8<GT>(p, tmk, tmv, it, dc, ctl, ps, wc);
  } else if constexpr (GT == 1) {
    decode_simt<GT, HD>(p, it, dc, ctl, ps, wc);
  } else {
    decode_tc<GT, HD>(p, tmk, tmv, it, dc, ctl, ps, wc);
  }
  named_bar_sync(dc.bar_id, dc.bar_threads);
  const float* scr = reinterpret_cast<const float*>(dc.ring);
  if (!ctl->abort) {
    const int nsplit = unit >= 0 ? p.units[unit * kUnitWords + 0] : 1;
    const int slot0 = unit >= 0 ? p.units[unit * kUnitWords + 1] : 0;
    float* slot = unit >= 0 ? p.partial_d + (size_t)(slot0 + split) * decode_slot_floats(G) : nullptr;
    for (int idx = ltid; idx < G * HD; idx += dc.bar_threads) {
      const int h = idx / HD, c = idx % HD;
      float mx = -INFINITY;
      for (int w = 0; w < dc.nw; ++w) mx = fmaxf(mx, scr[(w * GT + h) * kScr + kHeadDim]);
      float num = 0.f, den = 0.f;
      for (int w = 0; w < dc.nw; ++w) {
        const float* src = scr + (w * GT + h) * kScr;
        const float mw = src[kHeadDim];
        if (mw == -INFINITY) continue;
        const float f = ex2(mw - mx);
        num += f * src[c];
        den += f * src[kHeadDim + 1];
      }
      if (unit < 0) {
        p.o_decode[((size_t)d * p.Hq + (size_t)g * G + h) * HD + c] = f2bf(num / den);
      } else {
        slot[h * kRow + c] = num;
        if (c == 0) {
          slot[h * kRow + kHeadDim] = mx;
          slot[h * kRow + kHeadDim + 1] = den;
        }
      }
    }
    if (unit >= 0) {
      __threadfence();
      named_bar_sync(dc.bar_id, dc.bar_threads);
      if (ltid == 0) ctl->merge_last[dc.slot] = (atomicAdd(&p.arrive[unit], 1) == nsplit - 1);
      named_bar_sync(dc.bar_id, dc.bar_threads);
      if (ctl->merge_last[dc.slot]) {
        __threadfence();
        // the splits' (m, l) once into shared memory (the scratch is free again), one weight
        // per (head, split), then every output element as a weighted sum over the splits with
        // the loads of all of this thread's elements in flight together
        const size_t stride = (size_t)decode_slot_floats(G);
        const float* part0 = p.partial_d + (size_t)slot0 * stride;
        float* wts = reinterpret_cast<float*>(dc.ring);   // [G][nsplit]: m, then the weight
        float* ls = wts + kMaxGroup * kMaxDecodeSplits;    // [G][nsplit]: l
        float* inv = ls + kMaxGroup * kMaxDecodeSplits;    // [G]: 1 / merged l
        for (int idx = ltid; idx < G * nsplit; idx += dc.bar_threads) {
          const int h = idx / nsplit, k = idx - h * nsplit;
          const float* sl = part0 + (size_t)k * stride + h * kRow;
          wts[idx] = __ldcg(sl + kHeadDim);
          ls[idx] = __ldcg(sl + kHeadDim + 1);
        }
        named_bar_sync(dc.bar_id, dc.bar_threads);
        if (ltid < G) {
          float* w = wts + ltid * nsplit;
          const float* l = ls + ltid * nsplit;
          float mx = -INFINITY;
          for (int k = 0; k < nsplit; ++k) mx = fmaxf(mx, w[k]);
          float den = 0.f;
          for (int k = 0; k < nsplit; ++k) {
            const float f = w[k] == -INFINITY ? 0.f : ex2(w[k] - mx);
            w[k] = f;
            den += f * l[k];
          }
          inv[ltid] = 1.f / den;
        }
        named_bar_sync(dc.bar_id, dc.bar_threads);
        constexpr int kPer = (GT * HD + kDecodeWarps * 32 - 1) / (kDecodeWarps * 32);
        float num[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) num[e] = 0.f;
        for (int k = 0; k < nsplit; ++k) {
          const float* sl = part0 + (size_t)k * stride;
#pragma unroll
          for (int e = 0; e < kPer; ++e) {
            const int idx = ltid + e * kDecodeWarps * 32;
            if (idx < G * HD) {
              const int h = idx / HD, c = idx % HD;
              num[e] += wts[h * nsplit + k] * __ldcg(sl + h * kRow + c);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int idx = ltid + e * kDecodeWarps * 32;
          if (idx < G * HD) {
            const int h = idx / HD, c = idx % HD;
            p.o_decode[((size_t)d * p.Hq + (size_t)g * G + h) * HD + c] = f2bf(num[e] * inv[h]);
          }
        }
        if (ltid == 0) p.arrive[unit] = 0;
      }
    }
  }
  named_bar_sync(dc.bar_id, dc.bar_threads);
}

// ============================================================================ scheduler
// Next item for a slot. The prefill slot (0) of CTAs 0 .. max_prefill_ctas - 1 takes prefill
// tickets, and a decode ticket once the prefill list is drained (or in a decode-only launch, or
// on a CTA past the cap); the decode slot (1) and the prefill warps' two decode slots (2, 3) take
// decode tickets only. Per-SM counters record how many decode items each SM's prefill warps took
// over.
__device__ __forceinline__ void pick_item(const Params& p, int slot, int sm, SmemCtl* ctl) {
  int32_t* cnt = p.counters;
  int kind = -1, idx = 0;
  const bool may_prefill =
      slot == 0 && p.mode != kModeDecodeOnly && (int)blockIdx.x < p.max_prefill_ctas;
  const bool may_decode = p.mode != kModePrefillOnly;
  if (may_prefill) {
    const int t = atomicAdd(&cnt[0], 1);
    if (t < p.n_items_p) kind = 0, idx = t;
  }
  if (kind < 0 && may_decode) {
    const int t = atomicAdd(&cnt[1], 1);
    if (t < p.n_items_d) {
      kind = 1, idx = t;
      if (slot != 1) atomicAdd(&cnt[kCounterHeader + sm], 1);
    }
  }
  ctl->item_kind[slot] = kind;
  ctl->item_idx[slot] = idx;
}

__device__ __forceinline__ void record_item(const Params& p, int kind, int idx, uint32_t sm_raw,
                                            uint64_t t0) {
  pod_attn_item_record* rec = p.records + (kind == 0 ? idx : p.n_items_p + idx);
  rec->smid = (int32_t)sm_raw;
  rec->kind = kind;
  rec->item = idx;
  rec->cta = blockIdx.x;
  rec->t_start = t0;
  rec->t_end = globaltimer();
}

// A decode slot's ticket loop; `first` >= 0 is an item already taken for it.
template <int GT, int HD, bool FP8>
__device__ void decode_loop(const Params& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                            const DecodeCtx& dc, int first, int sm, uint32_t sm_raw, SmemCtl* ctl,
                            PipeState& ps, const WaitCtx& wc) {
  const bool leader = threadIdx.x == dc.first_thread;
  for (;;) {
    if (leader) {
      if (first >= 0) {
        ctl->item_kind[dc.slot] = 1;
        ctl->item_idx[dc.slot] = first;
      } else {
        pick_item(p, dc.slot, sm, ctl);
      }
    }
    first = -1;
    named_bar_sync(dc.bar_id, dc.bar_threads);
    const int kind = ctl->item_kind[dc.slot], idx = ctl->item_idx[dc.slot];
    if (kind < 0 || ctl->abort) break;
    const uint64_t t0 = (p.records != nullptr && leader) ? globaltimer() : 0;
    decode_item<GT, HD, FP8>(p, tmk, tmv, p.items_d + (size_t)idx * kItemWords, dc, ctl, ps, wc);
    if (p.records != nullptr && leader) record_item(p, kind, idx, sm_raw, t0);
  }
}

template <int GT, int HD, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    pod_attn_kernel(const __grid_constant__ Params p,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmkb,
                    const __grid_constant__ CUtensorMap tmvb) {
  extern __shared__ __align__(1024) uint8_t smem[];
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + kSmemCtlOff);
  if (smem_u32(smem) & 1023u) {  // the 128-byte swizzle needs 1024-byte-aligned tiles
    if (threadIdx.x == 0) record_error(p.status, POD_ATTN_ERR_CUDA);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool use_tmem = p.mode != kModeDecodeOnly && p.n_items_p > 0;

  if (tid == 0) {
    mbar_init(smem_u32(&ctl->q_full), 8);
    for (int i = 0; i < kKVStages; ++i) {
      mbar_init(smem_u32(&ctl->kv_full[i]), 1);
      mbar_init(smem_u32(&ctl->kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->s_full[i]), 1);
      mbar_init(smem_u32(&ctl->p_ready[i]), 8);
    }
    mbar_init(smem_u32(&ctl->pv_done), 1);
    mbar_init(smem_u32(&ctl->o_done), 1);
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < kDecodeSlotsFp8; ++s) mbar_init(smem_u32(&ctl->dslot[w][s]), 1);
    ctl->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    if (use_tmem) {
      prefetch_tmap(&tmkb);
      prefetch_tmap(&tmvb);
    }
  }
  if (use_tmem && warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const WaitCtx wc{&ctl->abort, p.status, p.timeout_ns};
  PipeState ps;
  if (p.n_new > 0) {
    // this CTA's share of the KV append, then one arrival; readers of appended rows wait for all
    append_rows<HD>(p);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(&p.counters[3], 1);
    }
  }
  const uint32_t sm_raw = smid();
  const int sm = (int)(sm_raw % (uint32_t)p.num_sms);
  if (warp < kDecodeWarp0) {
    // ------------------------------------------------------------------ prefill slot
    int handoff = -1;  // a decode item taken once the prefill list ran dry
    for (;;) {
      if (tid == 0) pick_item(p, 0, sm, ctl);
      named_bar_sync(1, kPrefillThreads);
      const int kind = ctl->item_kind[0], idx = ctl->item_idx[0];
      if (kind < 0 || ctl->abort) break;
      if (kind == 1) {
        handoff = idx;
        break;
      }
      const uint64_t t0 = (p.records != nullptr && tid == 0) ? globaltimer() : 0;
      if constexpr (!FP8)
        prefill_item<HD>(p, &tmk, &tmv, &tmkb, &tmvb, p.items_p + (size_t)idx * kItemWords, smem, ctl,
                         ps, wc);
      if (p.records != nullptr && tid == 0) record_item(p, kind, idx, sm_raw, t0);
    }
    if (handoff >= 0 && FP8) {
      // FP8 cache decode: warps 4-7, 8-11 and 0-3 become three 4-warp decode slots (the
      // producer and issuer warps have no prefill work here), each with a region of
      // kFp8GroupBytes (the decode slot's is the fourth)
      const int sub = warp >= kSoftmaxWarp0 ? (warp - kSoftmaxWarp0) / kDecodeWarps : 2;
      const int w0 = (warp / kDecodeWarps) * kDecodeWarps;
      const int grp = w0 / kDecodeWarps;
      const DecodeCtx dc{w0, kDecodeWarps, smem + grp * kFp8GroupBytes,
                         reinterpret_cast<float*>(smem + kFp8Groups * kFp8GroupBytes +
                                                  grp * kDecodeWarps * kSmemScoresPerWarp),
                         4 + sub, kDecodeWarps * 32, w0 * 32, 2 + sub};
      decode_loop<GT, HD, FP8>(p, &tmk, &tmv, dc, sub == 0 ? handoff : -1, sm, sm_raw, ctl, ps,
                               wc);
    } else if (handoff >= 0 && warp >= kSoftmaxWarp0) {
      // the softmax warps become two 4-warp decode slots over the prefill region
      const int sub = (warp - kSoftmaxWarp0) / kDecodeWarps;
      const int w0 = kSoftmaxWarp0 + sub * kDecodeWarps;
      const DecodeCtx dc{w0, kDecodeWarps, smem + sub * kSmemDecodeRing,
                         reinterpret_cast<float*>(smem + 2 * kSmemDecodeRing +
                                                  sub * kDecodeWarps * kSmemScoresPerWarp),
                         4 + sub, kDecodeWarps * 32, w0 * 32, 2 + sub};
      decode_loop<GT, HD, FP8>(p, &tmk, &tmv, dc, sub == 0 ? handoff : -1, sm, sm_raw, ctl, ps,
                               wc);
    }
  } else {
    // ------------------------------------------------------------------ decode slot
    const int ring_off = FP8 ? 3 * kFp8GroupBytes : kSmemDecodeOff;
    const int scores_off =
        FP8 ? kFp8Groups * kFp8GroupBytes + 3 * kDecodeWarps * kSmemScoresPerWarp : kSmemScoresOff;
    const DecodeCtx dc{kDecodeWarp0, kDecodeWarps, smem + ring_off,
                       reinterpret_cast<float*>(smem + scores_off), 3, kDecodeWarps * 32,
                       kDecodeWarp0 * 32, 1};
    decode_loop<GT, HD, FP8>(p, &tmk, &tmv, dc, -1, sm, sm_raw, ctl, ps, wc);
  }
  tc_fence_before();
  __syncthreads();
  if (ctl->abort && tid == 0) {
    // give copies still in flight time to land before this CTA's shared memory is released
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
  }
  __syncthreads();
  tc_fence_after();
  if (use_tmem && warp == 1) tmem_dealloc(ctl->tmem_base, kTmemCols);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.counters[2], 1) == (int)gridDim.x - 1) {
      p.counters[0] = 0;
      p.counters[1] = 0;
      p.counters[2] = 0;
      p.counters[3] = 0;
      __threadfence();
    }
  }
}

__global__ void selftest_timeout_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, status, timeout_ns};
    mbar_wait(smem_u32(&bar), 0, wc);  // nobody arrives: runs into the time limit
  }
}

// ============================================================================ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct CudaState {
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  CUtensorMap tmk{}, tmv{}, tmkb{}, tmvb{};
  const void *kk = nullptr, *kv = nullptr;  // pointers the maps were built for
  CUtensorMap tmk8{}, tmv8{};                               // e4m3 pools (FP8 cache decode)
  const void *kk8 = nullptr, *kv8 = nullptr;
};

// K or V pool: 2-D {dim, row} over num_blocks*Hkv*16 rows; one box is one paged block's 16 rows
// x 64 dims.
static bool encode_pool(CUtensorMap* m, const void* pool, int64_t rows, int hd) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kBlockSize};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V pool (head dim 128) seen per paged block: 3-D {64 dims, row, 64-dim half} with the half
// (128 bytes apart) as the outermost coordinate, so one box {64, 16, 2} is a block's 16 rows of
// both halves, landing half by half ([half][row][64 dims]).
static bool encode_pool_blocks(CUtensorMap* m, const void* pool, int64_t rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kBlockSize, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K pool (head dim 128) seen per paged block for the prefill tiles: 4-D {64 dims, row within an
// 8-row group, 64-dim half, 8-row group} (strides 256, 128 and 2048 bytes), so one box
// {64, 8, 2, 2} is a block's 16 rows of both halves, landing as [group][half][8 rows][64 dims].
static bool encode_pool_kblocks(CUtensorMap* m, const void* pool, int64_t rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, 128, (cuuint64_t)kHeadDim * 2 * 8};
  cuuint32_t box[4] = {64, 8, 2, 2};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 K or V pool: 2-D {byte, row}; one box is one paged block's 16 rows x 128 bytes.
static bool encode_pool8(CUtensorMap* m, const void* pool, int64_t rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)kBlockSize};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int GT, int HD, bool FP8 = false>
static cudaError_t launch_mode(const Params& p, int grid, cudaStream_t st, const CudaState& cs) {
  const CUtensorMap& tmk = FP8 ? cs.tmk8 : cs.tmk;
  const CUtensorMap& tmv = FP8 ? cs.tmv8 : cs.tmv;
  static std::atomic<int> attr_set{0};
  if (!attr_set.load()) {
    cudaError_t e = cudaFuncSetAttribute(pod_attn_kernel<GT, HD, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  if (!p.wait_append) {
    pod_attn_kernel<GT, HD, FP8><<<grid, kThreads, kSmemTotal, st>>>(p, tmk, tmv, cs.tmkb,
                                                                     cs.tmvb);
    return cudaGetLastError();
  }
  // Items wait for every CTA's share of the append: a cooperative launch guarantees that all
  // CTAs are resident at once (or fails to launch), so the wait cannot starve.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemTotal;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pod_attn_kernel<GT, HD, FP8>, p, tmk, tmv, cs.tmkb,
                            cs.tmvb);
}

template <int HD>
static cudaError_t launch_hd(const Params& p, int grid, cudaStream_t st, const CudaState& cs) {
  switch (p.G) {
    case 1: return launch_mode<1, HD>(p, grid, st, cs);
    case 2: return launch_mode<2, HD>(p, grid, st, cs);
    case 3:
    case 4: return launch_mode<4, HD>(p, grid, st, cs);
    default: return launch_mode<8, HD>(p, grid, st, cs);
  }
}

static cudaError_t launch(const Params& p, int grid, cudaStream_t st, const CudaState& cs) {
  if (grid <= 0) return cudaSuccess;
  return p.head_dim == 64 ? launch_hd<64>(p, grid, st, cs) : launch_hd<128>(p, grid, st, cs);
}

// The FP8-cache decode launch (head dim 128).
static cudaError_t launch_fp8(const Params& p, int grid, cudaStream_t st, const CudaState& cs) {
  if (grid <= 0) return cudaSuccess;
  switch (p.G) {
    case 1: return launch_mode<1, 128, true>(p, grid, st, cs);
    case 2: return launch_mode<2, 128, true>(p, grid, st, cs);
    case 3:
    case 4: return launch_mode<4, 128, true>(p, grid, st, cs);
    default: return launch_mode<8, 128, true>(p, grid, st, cs);
  }
}

// ---------------------------------------------------------------- allocation-free scratch
// The workspace of pod_attn_run_static: one array per device that loads this library, alive
// until the process exits. Host code must not use the symbol's name as an address (it is a host
// stand-in); static_scratch() looks up its device address per device.
constexpr size_t kStaticScratchBytes = POD_ATTN_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

static pod_attn_status static_scratch(void** out) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return POD_ATTN_ERR_CUDA;
    }
    addr[dev] = ptr;
  }
  *out = addr[dev];
  return POD_ATTN_OK;
}

}  // namespace pod

using namespace pod;

// ============================================================================ C ABI
extern "C" {

const char* pod_attn_status_string(pod_attn_status s) {
  switch (s) {
    case POD_ATTN_OK: return "ok";
    case POD_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case POD_ATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case POD_ATTN_ERR_WORKSPACE: return "workspace too small or misaligned";
    case POD_ATTN_ERR_CUDA: return "CUDA error";
    case POD_ATTN_ERR_BAD_INDEX: return "block-table entry out of range";
    case POD_ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

pod_attn_status pod_attn_plan(const pod_attn_problem* problem, const int32_t* h_cu_seqlens_q,
                              const int32_t* h_kv_lens, const pod_attn_options* options,
                              pod_attn_plan_t* out) {
  if (problem == nullptr || out == nullptr) return POD_ATTN_ERR_INVALID_ARG;
  *out = nullptr;
  pod_attn_options opt{};
  if (options) opt = *options;
  if (opt.variant != POD_ATTN_FUSED && opt.variant != POD_ATTN_SERIAL &&
      opt.variant != POD_ATTN_STREAMS)
    return POD_ATTN_ERR_INVALID_ARG;
  int num_sms = opt.num_sms;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return POD_ATTN_ERR_CUDA;
    }
  }
  pod_attn_plan_s* plan = new (std::nothrow) pod_attn_plan_s();
  if (!plan) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_status st;
  try {
    st = build_plan(*problem, h_cu_seqlens_q, h_kv_lens, opt, num_sms, plan);
  } catch (...) {
    st = POD_ATTN_ERR_INVALID_ARG;
  }
  if (st != POD_ATTN_OK) {
    delete plan;
    return st;
  }
  CudaState* cs = new (std::nothrow) CudaState();
  if (!cs) {
    delete plan;
    return POD_ATTN_ERR_INVALID_ARG;
  }
  if (opt.variant == POD_ATTN_STREAMS) {
    if (cudaEventCreateWithFlags(&cs->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&cs->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();  // tolerated here; run() reports it
      cs->ev_fork = cs->ev_join = nullptr;
    }
  }
  plan->cuda_state = cs;
  *out = plan;
  return POD_ATTN_OK;
}

size_t pod_attn_workspace_bytes(pod_attn_plan_t plan) { return plan ? plan->ws.total : 0; }

pod_attn_status pod_attn_plan_bucket(pod_attn_plan_t plan, pod_attn_bucket* out) {
  if (!plan || !out) return POD_ATTN_ERR_INVALID_ARG;
  const pod_attn_problem& pr = plan->prob;
  const int Np = pr.num_prefill_seqs, Nd = pr.num_decode_seqs;
  const int64_t hd = pr.head_dim;
  const int64_t row = 4 * hd;  // K + V (or q + o) of one row, bf16
  int64_t flops = 0, bytes = 0;
  for (int s = 0; s < Np; ++s) {
    const int64_t q = plan->cu[s + 1] - plan->cu[s], L = plan->kv[s], P = L - q;
    flops += 4 * hd * (int64_t)pr.num_q_heads *
             (plan->opt.non_causal == 0 ? q * P + q * (q + 1) / 2 : q * L);
    bytes += L * pr.num_kv_heads * row + q * pr.num_q_heads * row;
  }
  for (int d = 0; d < Nd; ++d)
    bytes += (int64_t)plan->kv[Np + d] * pr.num_kv_heads * row + (int64_t)pr.num_q_heads * row;
  auto bit_length = [](int64_t x) { int b = 0; while (x > 0) { ++b; x >>= 1; } return b; };
  auto bucket = [&](int64_t x, int64_t unit) { return x > 0 ? bit_length((x + unit - 1) / unit) : 0; };
  pod_attn_bucket r{};
  r.prefill_flops = flops;
  r.read_bytes = bytes;
  r.prefill_ctas = (int32_t)(plan->items_p.size() / kItemWords);
  r.decode_ctas = (int32_t)(plan->items_d.size() / kItemWords);
  r.grid = plan->grid_fused;
  r.smem_per_cta = kSmemTotal;
  r.tmem_cols_per_cta = r.prefill_ctas > 0 ? kTmemCols : 0;
  r.bucket_flops = bucket(flops, int64_t(1) << 30);
  r.bucket_bytes = bucket(bytes, int64_t(1) << 20);
  r.bucket_ctas = bit_length((int64_t)r.prefill_ctas + r.decode_ctas);
  r.intensity = bytes > 0 ? (double)flops / (double)bytes : 0.0;
  *out = r;
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_get_plan_info(pod_attn_plan_t plan, pod_attn_plan_info* info) {
  if (!plan || !info) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_plan_info r{};
  r.num_prefill_items = (int32_t)(plan->items_p.size() / kItemWords);
  r.num_decode_items = (int32_t)(plan->items_d.size() / kItemWords);
  r.num_units = (int32_t)(plan->units.size() / kUnitWords);
  r.num_sms = plan->num_sms;
  r.ctas_per_sm = plan->ctas_per_sm;
  r.max_prefill_ctas = plan->max_prefill_ctas;
  r.grid_fused = plan->grid_fused;
  r.grid_prefill = plan->grid_prefill;
  r.grid_decode = plan->grid_decode;
  r.smem_bytes = kSmemTotal;
  r.threads_per_cta = kThreads;
  r.item_words = kItemWords;
  r.workspace_bytes = plan->ws.total;
  r.est_prefill_flops = plan->est_prefill_flops;
  r.est_prefill_bytes = plan->est_prefill_bytes;
  r.est_decode_bytes = plan->est_decode_bytes;
  r.est_decode_flops = plan->est_decode_flops;
  *info = r;
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_plan_items(pod_attn_plan_t plan, int32_t* out, size_t capacity,
                                    size_t* count) {
  if (!plan || !count) return POD_ATTN_ERR_INVALID_ARG;
  const size_t n = plan->items_p.size() + plan->items_d.size() + plan->units.size();
  *count = n;
  if (n == 0 || out == nullptr) return POD_ATTN_OK;  // size query
  if (capacity < n) return POD_ATTN_ERR_INVALID_ARG;
  std::memcpy(out, plan->items_p.data(), plan->items_p.size() * 4);
  std::memcpy(out + plan->items_p.size(), plan->items_d.data(), plan->items_d.size() * 4);
  std::memcpy(out + plan->items_p.size() + plan->items_d.size(), plan->units.data(),
              plan->units.size() * 4);
  return POD_ATTN_OK;
}

static pod_attn_status check_ws(pod_attn_plan_t plan, const void* ws, size_t bytes) {
  if (!ws) return POD_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0 || bytes < plan->ws.total)
    return POD_ATTN_ERR_WORKSPACE;
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_upload(pod_attn_plan_t plan, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!plan) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_status st = check_ws(plan, workspace, workspace_bytes);
  if (st != POD_ATTN_OK) return st;
  // one copy: the zeroed status, counters and arrival counters, then the work lists, laid out
  // on the host as they sit in the workspace
  const bool ok = plan->upload_image.empty() ||
                  cudaMemcpyAsync(workspace, plan->upload_image.data(), plan->upload_image.size(),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) ==
                      cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  return POD_ATTN_OK;
}

}  // extern "C"

// pod_attn_run and pod_attn_run_append; k_new == nullptr: no append.
static pod_attn_status run_impl(pod_attn_plan_t plan, const void* q_prefill, const void* q_decode,
                                const void* k_new, const void* v_new, const void* k_pool,
                                const void* v_pool, const int32_t* d_block_tables,
                                const int32_t* d_cu_seqlens_q, const int32_t* d_kv_lens,
                                void* o_prefill, void* o_decode, void* workspace,
                                size_t workspace_bytes, void* stream, void* stream2) {
  if (!plan) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_status st = check_ws(plan, workspace, workspace_bytes);
  if (st != POD_ATTN_OK) return st;
  if (plan->opt.kv_fp8) return POD_ATTN_ERR_UNSUPPORTED;  // a plan for the e4m3 cache
  const pod_attn_problem& pr = plan->prob;
  const int n_p = (int)(plan->items_p.size() / kItemWords);
  const int n_d = (int)(plan->items_d.size() / kItemWords);
  if (n_p + n_d == 0) return POD_ATTN_OK;
  if (!k_pool || !v_pool || !d_block_tables || !d_kv_lens) return POD_ATTN_ERR_INVALID_ARG;
  if (n_p > 0 && (!q_prefill || !o_prefill || !d_cu_seqlens_q)) return POD_ATTN_ERR_INVALID_ARG;
  if (n_d > 0 && (!q_decode || !o_decode)) return POD_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
       reinterpret_cast<uintptr_t>(q_prefill) | reinterpret_cast<uintptr_t>(o_prefill) |
       reinterpret_cast<uintptr_t>(q_decode) | reinterpret_cast<uintptr_t>(k_new) |
       reinterpret_cast<uintptr_t>(v_new)) & 15)
    return POD_ATTN_ERR_INVALID_ARG;
  CudaState* cs = static_cast<CudaState*>(plan->cuda_state);
  const int64_t pool_rows = (int64_t)pr.num_blocks * pr.num_kv_heads * kBlockSize;
  // the pools' maps serve the prefill tiles and the grouped-query decode path
  if (cs->kk != k_pool) {
    if (!encode_pool(&cs->tmk, k_pool, pool_rows, pr.head_dim)) return POD_ATTN_ERR_CUDA;
    // the prefill tiles' per-block view (head dim 128; a 64-dim head uses the 2-D map)
    if (pr.head_dim == kHeadDim ? !encode_pool_kblocks(&cs->tmkb, k_pool, pool_rows)
                                : !encode_pool(&cs->tmkb, k_pool, pool_rows, pr.head_dim))
      return POD_ATTN_ERR_CUDA;
    cs->kk = k_pool;
  }
  if (cs->kv != v_pool) {
    if (!encode_pool(&cs->tmv, v_pool, pool_rows, pr.head_dim)) return POD_ATTN_ERR_CUDA;
    // the prefill tiles' per-block view (head dim 128; a 64-dim head uses the 2-D map)
    if (pr.head_dim == kHeadDim ? !encode_pool_blocks(&cs->tmvb, v_pool, pool_rows)
                                : !encode_pool(&cs->tmvb, v_pool, pool_rows, pr.head_dim))
      return POD_ATTN_ERR_CUDA;
    cs->kv = v_pool;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const WorkspaceLayout& w = plan->ws;
  Params p{};
  p.q_prefill = static_cast<const uint16_t*>(q_prefill);
  p.q_decode = static_cast<const uint16_t*>(q_decode);
  p.k_pool = static_cast<const uint16_t*>(k_pool);
  p.v_pool = static_cast<const uint16_t*>(v_pool);
  p.block_tables = d_block_tables;
  p.cu_seqlens = d_cu_seqlens_q;
  p.kv_lens = d_kv_lens;
  p.o_prefill = static_cast<uint16_t*>(o_prefill);
  p.o_decode = static_cast<uint16_t*>(o_decode);
  p.items_p = reinterpret_cast<const int32_t*>(ws + w.items_p);
  p.items_d = reinterpret_cast<const int32_t*>(ws + w.items_d);
  p.units = reinterpret_cast<const int32_t*>(ws + w.units);
  p.partial_p = reinterpret_cast<float*>(ws + w.partial_p);
  p.partial_d = reinterpret_cast<float*>(ws + w.partial_d);
  p.arrive = reinterpret_cast<int32_t*>(ws + w.arrive);
  p.status = reinterpret_cast<int32_t*>(ws + w.status);
  p.records = plan->opt.instrument ? reinterpret_cast<pod_attn_item_record*>(ws + w.records) : nullptr;
  p.n_items_p = n_p;
  p.n_items_d = n_d;
  p.Hq = pr.num_q_heads;
  p.Hkv = pr.num_kv_heads;
  p.G = plan->group;
  p.Np = pr.num_prefill_seqs;
  p.Nd = pr.num_decode_seqs;
  p.num_blocks = pr.num_blocks;
  p.maxb = pr.max_blocks_per_seq;
  p.pool_rows = (int32_t)pool_rows;
  p.num_sms = plan->num_sms;
  p.max_prefill_ctas = plan->max_prefill_ctas;
  p.hp_log2 = __builtin_ctz((unsigned)plan->head_pack);
  p.causal = plan->opt.non_causal == 0;
  p.head_dim = pr.head_dim;
  p.tq = plan->tile_tokens;
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  p.timeout_ns = kWaitTimeoutNs;
  int32_t* counters = reinterpret_cast<int32_t*>(ws + w.counters);
  auto counter_block = [&](int mode) { return counters + (size_t)mode * w.counter_block_words; };
  const bool append = k_new != nullptr;
  const int n_new = (int)(plan->new_rows.size() / 2);
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_pool_w = static_cast<uint16_t*>(const_cast<void*>(k_pool));
  p.v_pool_w = static_cast<uint16_t*>(const_cast<void*>(v_pool));
  p.new_rows = reinterpret_cast<const int32_t*>(ws + w.new_rows);
  p.n_new = 0;
  p.new_first = 0;
  p.wait_append = 0;
  // SERIAL and STREAMS: the append runs as a launch of its own, ahead of both kinds of items
  Params ap = p;
  ap.mode = kModeAppendOnly;
  ap.counters = counter_block(kModeAppendOnly);
  ap.n_items_p = ap.n_items_d = 0;
  ap.n_new = n_new;
  const int grid_append =
      std::max(1, std::min(plan->num_sms, (n_new * pr.num_kv_heads + kWarps - 1) / kWarps));

  cudaStream_t s1 = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  switch (plan->opt.variant) {
    case POD_ATTN_FUSED: {
      p.mode = kModeFused;
      p.counters = counter_block(kModeFused);
      if (append) {  // in the same launch, ahead of the items that read the new rows
        p.n_new = n_new;
        p.wait_append = 1;
      }
      e = launch(p, plan->grid_fused, s1, *cs);
      break;
    }
    case POD_ATTN_SERIAL: {
      Params a = p, b = p;
      a.mode = kModePrefillOnly;
      a.counters = counter_block(kModePrefillOnly);
      b.mode = kModeDecodeOnly;
      b.counters = counter_block(kModeDecodeOnly);
      if (append && n_new > 0) e = launch(ap, grid_append, s1, *cs);
      if (e == cudaSuccess) e = launch(a, plan->grid_prefill, s1, *cs);
      if (e == cudaSuccess) e = launch(b, plan->grid_decode, s1, *cs);
      break;
    }
    case POD_ATTN_STREAMS: {
      if (!cs->ev_fork || !cs->ev_join) return POD_ATTN_ERR_CUDA;
      cudaStream_t s2 = static_cast<cudaStream_t>(stream2);
      Params a = p, b = p;
      a.mode = kModePrefillOnly;
      a.counters = counter_block(kModePrefillOnly);
      b.mode = kModeDecodeOnly;
      b.counters = counter_block(kModeDecodeOnly);
      if (append && n_new > 0) e = launch(ap, grid_append, s1, *cs);
      if (e == cudaSuccess) e = cudaEventRecord(cs->ev_fork, s1);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s2, cs->ev_fork, 0);
      if (e == cudaSuccess) e = launch(a, plan->grid_prefill, s1, *cs);
      if (e == cudaSuccess) e = launch(b, plan->grid_decode, s2, *cs);
      if (e == cudaSuccess) e = cudaEventRecord(cs->ev_join, s2);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s1, cs->ev_join, 0);
      break;
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  return POD_ATTN_OK;
}

extern "C" {

pod_attn_status pod_attn_run(pod_attn_plan_t plan, const void* q_prefill, const void* q_decode,
                             const void* k_pool, const void* v_pool,
                             const int32_t* d_block_tables, const int32_t* d_cu_seqlens_q,
                             const int32_t* d_kv_lens, void* o_prefill, void* o_decode,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* stream2) {
  return run_impl(plan, q_prefill, q_decode, nullptr, nullptr, k_pool, v_pool, d_block_tables,
                  d_cu_seqlens_q, d_kv_lens, o_prefill, o_decode, workspace, workspace_bytes,
                  stream, stream2);
}

pod_attn_status pod_attn_run_append(pod_attn_plan_t plan, const void* q_prefill,
                                    const void* q_decode, const void* k_new, const void* v_new,
                                    void* k_pool, void* v_pool, const int32_t* d_block_tables,
                                    const int32_t* d_cu_seqlens_q, const int32_t* d_kv_lens,
                                    void* o_prefill, void* o_decode, void* workspace,
                                    size_t workspace_bytes, void* stream, void* stream2) {
  if (!k_new || !v_new) return POD_ATTN_ERR_INVALID_ARG;
  return run_impl(plan, q_prefill, q_decode, k_new, v_new, k_pool, v_pool, d_block_tables,
                  d_cu_seqlens_q, d_kv_lens, o_prefill, o_decode, workspace, workspace_bytes,
                  stream, stream2);
}

pod_attn_status pod_attn_run_decode_fp8(pod_attn_plan_t plan, const void* q_decode,
                                        const void* k_pool8, const void* v_pool8,
                                        const float* d_k_scale, const float* d_v_scale,
                                        const int32_t* d_block_tables, const int32_t* d_kv_lens,
                                        void* o_decode, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (!plan) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_status st = check_ws(plan, workspace, workspace_bytes);
  if (st != POD_ATTN_OK) return st;
  const pod_attn_problem& pr = plan->prob;
  if (!plan->opt.kv_fp8 || pr.num_prefill_seqs != 0 || pr.head_dim != kHeadDim)
    return POD_ATTN_ERR_UNSUPPORTED;
  const int n_d = (int)(plan->items_d.size() / kItemWords);
  if (n_d == 0) return POD_ATTN_OK;
  if (!q_decode || !o_decode || !k_pool8 || !v_pool8 || !d_k_scale || !d_v_scale ||
      !d_block_tables || !d_kv_lens)
    return POD_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_decode) | reinterpret_cast<uintptr_t>(o_decode) |
       reinterpret_cast<uintptr_t>(k_pool8) | reinterpret_cast<uintptr_t>(v_pool8) |
       reinterpret_cast<uintptr_t>(d_k_scale) | reinterpret_cast<uintptr_t>(d_v_scale)) & 15)
    return POD_ATTN_ERR_INVALID_ARG;
  CudaState* cs = static_cast<CudaState*>(plan->cuda_state);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const WorkspaceLayout& w = plan->ws;
  Params p{};
  p.q_decode = static_cast<const uint16_t*>(q_decode);
  p.o_decode = static_cast<uint16_t*>(o_decode);
  p.k8 = static_cast<const uint8_t*>(k_pool8);
  p.v8 = static_cast<const uint8_t*>(v_pool8);
  p.k_scale = d_k_scale;
  p.v_scale = d_v_scale;
  p.block_tables = d_block_tables;
  p.kv_lens = d_kv_lens;
  p.items_p = reinterpret_cast<const int32_t*>(ws + w.items_p);
  p.items_d = reinterpret_cast<const int32_t*>(ws + w.items_d);
  p.units = reinterpret_cast<const int32_t*>(ws + w.units);
  p.partial_p = reinterpret_cast<float*>(ws + w.partial_p);
  p.partial_d = reinterpret_cast<float*>(ws + w.partial_d);
  p.arrive = reinterpret_cast<int32_t*>(ws + w.arrive);
  p.status = reinterpret_cast<int32_t*>(ws + w.status);
  p.records = plan->opt.instrument ? reinterpret_cast<pod_attn_item_record*>(ws + w.records) : nullptr;
  p.n_items_p = 0;
  p.n_items_d = n_d;
  p.Hq = pr.num_q_heads;
  p.Hkv = pr.num_kv_heads;
  p.G = plan->group;
  p.Np = 0;
  p.Nd = pr.num_decode_seqs;
  p.num_blocks = pr.num_blocks;
  p.maxb = pr.max_blocks_per_seq;
  p.pool_rows = (int32_t)((int64_t)pr.num_blocks * pr.num_kv_heads * kBlockSize);
  p.num_sms = plan->num_sms;
  p.max_prefill_ctas = 0;
  p.hp_log2 = 0;
  p.tq = kTileM;
  p.causal = 1;
  p.head_dim = kHeadDim;
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  p.timeout_ns = kWaitTimeoutNs;
  p.mode = kModeFused;
  p.counters = reinterpret_cast<int32_t*>(ws + w.counters);  // the fused launch's block
  if (cs->kk8 != k_pool8) {
    if (!encode_pool8(&cs->tmk8, k_pool8, p.pool_rows)) return POD_ATTN_ERR_CUDA;
    cs->kk8 = k_pool8;
  }
  if (cs->kv8 != v_pool8) {
    if (!encode_pool8(&cs->tmv8, v_pool8, p.pool_rows)) return POD_ATTN_ERR_CUDA;
    cs->kv8 = v_pool8;
  }
  const cudaError_t e = launch_fp8(p, plan->grid_fused, static_cast<cudaStream_t>(stream), *cs);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_append_fp8(pod_attn_plan_t plan, const void* k_new, const void* v_new,
                                    void* k_pool8, void* v_pool8, const float* d_k_scale,
                                    float* d_v_scale, const int32_t* d_block_tables,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan) return POD_ATTN_ERR_INVALID_ARG;
  pod_attn_status st = check_ws(plan, workspace, workspace_bytes);
  if (st != POD_ATTN_OK) return st;
  const pod_attn_problem& pr = plan->prob;
  if (!plan->opt.kv_fp8 || pr.num_prefill_seqs != 0 || pr.head_dim != kHeadDim)
    return POD_ATTN_ERR_UNSUPPORTED;
  const int n_new = pr.num_decode_seqs;
  if (n_new == 0) return POD_ATTN_OK;
  if (!k_new || !v_new || !k_pool8 || !v_pool8 || !d_k_scale || !d_v_scale || !d_block_tables)
    return POD_ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_pool8) | reinterpret_cast<uintptr_t>(v_pool8) |
       reinterpret_cast<uintptr_t>(d_k_scale) | reinterpret_cast<uintptr_t>(d_v_scale)) & 15)
    return POD_ATTN_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AppendFp8Args a{};
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k8 = static_cast<uint8_t*>(k_pool8);
  a.v8 = static_cast<uint8_t*>(v_pool8);
  a.k_scale = d_k_scale;
  a.v_scale = d_v_scale;
  a.block_tables = d_block_tables;
  a.new_rows = reinterpret_cast<const int32_t*>(ws + plan->ws.new_rows);
  a.status = reinterpret_cast<int32_t*>(ws + plan->ws.status);
  a.n_new = n_new;
  a.Hkv = pr.num_kv_heads;
  a.maxb = pr.max_blocks_per_seq;
  a.num_blocks = pr.num_blocks;
  const int units = n_new * pr.num_kv_heads;
  const int grid = std::max(1, std::min(plan->num_sms * 4, (units + 7) / 8));
  append_fp8_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  if (cudaGetLastError() != cudaSuccess) return POD_ATTN_ERR_CUDA;
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_last_device_status(pod_attn_plan_t plan, void* workspace, void* stream) {
  (void)plan;
  if (!workspace) {  // the status word of pod_attn_run_static's scratch array on this device
    const pod_attn_status st = static_scratch(&workspace);
    if (st != POD_ATTN_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t code = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpy(&code, workspace, sizeof code, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(workspace, 0, sizeof code) != cudaSuccess) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  if (code == POD_ATTN_ERR_BAD_INDEX || code == POD_ATTN_ERR_TIMEOUT)
    return static_cast<pod_attn_status>(code);
  return code == 0 ? POD_ATTN_OK : POD_ATTN_ERR_CUDA;
}

pod_attn_status pod_attn_read_records(pod_attn_plan_t plan, const void* workspace,
                                      pod_attn_item_record* out, size_t capacity, size_t* count,
                                      void* stream) {
  if (!plan || !workspace || !count || !plan->opt.instrument) return POD_ATTN_ERR_INVALID_ARG;
  const size_t n = plan->items_p.size() / kItemWords + plan->items_d.size() / kItemWords;
  *count = n;
  if (n == 0) return POD_ATTN_OK;
  if (!out || capacity < n) return POD_ATTN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(out, static_cast<const uint8_t*>(workspace) + plan->ws.records,
                 n * sizeof(pod_attn_item_record), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return POD_ATTN_ERR_CUDA;
  }
  return POD_ATTN_OK;
}

pod_attn_status pod_attn_run_static(pod_attn_plan_t plan, const void* q_prefill,
                                    const void* q_decode, const void* k_pool,
                                    const void* v_pool, const int32_t* d_block_tables,
                                    const int32_t* d_cu_seqlens_q, const int32_t* d_kv_lens,
                                    void* o_prefill, void* o_decode, void* stream) {
  // instrumentation records would land in the shared array, where no caller can read them
  if (!plan || plan->opt.variant != POD_ATTN_FUSED || plan->opt.instrument)
    return POD_ATTN_ERR_INVALID_ARG;
  if (plan->opt.kv_fp8) return POD_ATTN_ERR_UNSUPPORTED;
  if (plan->ws.total > kStaticScratchBytes) return POD_ATTN_ERR_WORKSPACE;
  {
    // the array's address is the current device's: the stream must belong to that device
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
      cudaGetLastError();
      return POD_ATTN_ERR_CUDA;
    }
    if (sdev != cur) return POD_ATTN_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  pod_attn_status st = static_scratch(&scratch);
  if (st != POD_ATTN_OK) return st;
  // work lists in, status / scheduling / merge counters cleared: the array keeps the last
  // call's contents
  st = pod_attn_upload(plan, scratch, kStaticScratchBytes, stream);
  if (st != POD_ATTN_OK) return st;
  return pod_attn_run(plan, q_prefill, q_decode, k_pool, v_pool, d_block_tables,
                      d_cu_seqlens_q, d_kv_lens, o_prefill, o_decode, scratch,
                      kStaticScratchBytes, stream, nullptr);
}

void pod_attn_plan_destroy(pod_attn_plan_t plan) {
  if (!plan) return;
  CudaState* cs = static_cast<CudaState*>(plan->cuda_state);
  if (cs) {
    if (cs->ev_fork) cudaEventDestroy(cs->ev_fork);
    if (cs->ev_join) cudaEventDestroy(cs->ev_join);
    delete cs;
  }
  delete plan;
}

pod_attn_status pod_attn_selftest_timeout(void* workspace, int32_t timeout_us, void* stream) {
  if (!workspace || timeout_us < 1) return POD_ATTN_ERR_INVALID_ARG;
  selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(workspace), (uint64_t)timeout_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return POD_ATTN_ERR_CUDA;
  return POD_ATTN_OK;
}

}  // extern "C"
