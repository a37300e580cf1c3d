// planner.cpp — host planner of the hybrid prefill+decode launch.
//
// "POD-Attention" digest (Silicon & Systems), §"가상 CTA와 SM별 균형": a normal grid of CTAs
// is mapped onto virtual prefill and decode CTAs; the number of CTAs one prefill chunk may
// generate is limited so decode work is not pushed out. §"동시 실행만으로 부족한 이유": a CTA
// count just above a multiple of what the SMs hold at once costs a whole extra wave.
//
// This file turns one hybrid batch into two work lists (virtual CTAs):
//   prefill item = (chunk s, tile t, block of hp query heads, KV split k) — a tile is 128
//                  rows = 128/hp tokens x hp heads of one kv-head group
//   decode item  = (sequence d, kv-head g, KV split k)   — one item serves all G query heads
//                  of the kv-head (GQA grouping, "LLMSO - W4", §"KV 헤드 줄이기")
// and sizes the persistent grid: one CTA per SM, each with a prefill slot and a decode slot
// that pull items from the two lists.
//
// Split planning. Every item gets a cost (decode: 8 per 16-row K/V block, i.e. its bytes in
// KiB; prefill: 57 per 128-key step of its 128 rows, its tensor-core time expressed in the
// same byte-time units at a 6.8 TB/s : 1 PFLOP/s balance). Outputs are split along the keys
// ("LLMSO - W4", §"FlashDecoding — decode 단계의 병렬성 확보"), so no single item can leave a
// long tail after the others finish:
//  * prefill: one chunk size c (steps per item) for all outputs, c = ceil(longest / k) for
//    k = 1..8 (at least 4 steps), the one that minimises the makespan of the items taken
//    longest first by the SMs' prefill slots, each to the slot that frees first, with a fixed
//    per-item overhead. A split count just past a multiple of the SMs costs a whole extra
//    round of items (§"동시 실행만으로 부족한 이유"), which this model sees.
//  * decode: with W the total cost and S the item slots, an output whose cost exceeds
//    W / (4 S) is split into at most 64 parts of at least 12 blocks.
// Items are then ordered longest first. All arithmetic is integer, so the plan is reproducible
// bit for bit.
//
// Decode-only plans (no prefill work; the FP8-cache decode is one) know how many items run at
// once: S = groups x SMs 4-warp decode groups (3 per SM on a bf16 cache, where the prefill
// slot's softmax warps become two groups beside the decode slot; 4 on an e4m3 cache, where its
// producer and issuer warps become a third). There one chunk size c (blocks per item, before
// each output is rebalanced into equal parts) is chosen for all outputs to minimise the makespan of
// the items taken longest first by S groups, modelled wave by wave (each wave of S items lasts
// as long as its longest), each item costing ceil(blocks / 4) + 2 block-times of one warp (its
// four warps share the blocks; the 2 stand for its start and merge). A split count just past a multiple of S costs a whole extra wave
// of items (the wave-quantisation point of §"동시 실행만으로 부족한 이유"), which the
// W / (4 S) rule above cannot see.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>

#include "pod_internal.h"

namespace pod {
namespace {

constexpr int64_t kDecodeBlockCost = 8;   // 16 rows x (K + V) x 128 x bf16 = 8 KiB
constexpr int64_t kPrefillStepCost = 57;  // 4*128*128*128 FLOPs at the byte-time balance
constexpr int kMinDecodeBlocksPerSplit = 12;
constexpr int kMinPrefillTilesPerSplit = 4;
constexpr int64_t kPrefillItemOverhead = 8;  // per-item start and epilogue, in steps
constexpr int64_t kDecodeItemOverhead = 2;   // per-item start and merge, in warp block-times
constexpr int kDecodeGroupsBf16 = 3;         // 4-warp decode groups per SM, bf16 cache
constexpr int kDecodeGroupsFp8 = 4;          // ... e4m3 cache
// chunk candidates of the decode-only rule: ceil(longest output / k)
constexpr int kChunkDivisors[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 20, 24, 32, 40, 48, 64};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split of one output of `nblk` blocks for a chunk of about `c` blocks: ns parts of
// ceil(nblk / ns) blocks (the last one shorter).
inline void rebalanced(int64_t nblk, int64_t c, int64_t* ns, int64_t* chunk) {
  *ns = std::max<int64_t>(1, std::min(ceil_div(nblk, c), nblk));
  *chunk = ceil_div(nblk, *ns);
  *ns = ceil_div(nblk, *chunk);
}

// Modelled makespan (in warp block-times) of the items that chunk size c makes of the outputs
// `nblks` on `slots` decode groups taking them longest first: wave w holds the items ranked
// w*slots .. (w+1)*slots - 1 and lasts as long as its first (longest) one. Item costs are
// counted in `hist` (indexed by cost), so this is linear in the outputs and the largest cost.
int64_t decode_makespan(const std::vector<int64_t>& nblks, int64_t c, int64_t slots,
                        std::vector<int64_t>& hist) {
  std::fill(hist.begin(), hist.end(), 0);
  int64_t top = 0;
  for (int64_t n : nblks) {
    int64_t ns, ch;
    rebalanced(n, c, &ns, &ch);
    const int64_t full = ceil_div(ch, 4) + kDecodeItemOverhead;
    const int64_t last = ceil_div(n - (ns - 1) * ch, 4) + kDecodeItemOverhead;
    hist[full] += ns - 1;
    hist[last] += 1;
    top = std::max(top, full);
  }
  int64_t span = 0, rank = 0, next_head = 0;  // rank of the next item; rank of the next wave head
  for (int64_t x = top; x > 0; --x) {
    const int64_t k = hist[x];
    if (k == 0) continue;
    // wave heads among ranks [rank, rank + k)
    if (next_head < rank + k) {
      const int64_t heads = (rank + k - 1 - next_head) / slots + 1;
      span += heads * x;
      next_head += heads * slots;
    }
    rank += k;
  }
  return span;
}

// Modelled makespan (in steps) of the prefill items that chunk size c makes of the outputs
// `nts` on `slots` prefill slots taking them longest first, each to the slot that frees first
// (list scheduling); an item costs its steps plus kPrefillItemOverhead. The makespan depends
// only on the multiset of slot loads, so the items are counted by cost (`hist`) and the loads
// kept as a histogram (`load`): the least loaded slot's load never decreases, so a cursor
// finds it, and the whole model is linear in the items and the largest load.
int64_t prefill_makespan(const std::vector<int64_t>& nts, int64_t c, int64_t slots,
                         std::vector<int64_t>& hist, std::vector<int64_t>& load) {
  int64_t top = 0, total = 0;
  for (int64_t n : nts) top = std::max(top, std::min(c, n) + kPrefillItemOverhead);
  hist.assign((size_t)top + 1, 0);
  for (int64_t n : nts) {
    int64_t ns, ch;
    rebalanced(n, c, &ns, &ch);
    const int64_t last = n - (ns - 1) * ch + kPrefillItemOverhead;
    hist[(size_t)(ch + kPrefillItemOverhead)] += ns - 1;
    hist[(size_t)last] += 1;
    total += (ns - 1) * (ch + kPrefillItemOverhead) + last;
  }
  // an item starts at the least load, which is at most total / slots
  load.assign((size_t)(total / slots + top + 1), 0);
  load[0] = slots;
  int64_t cur = 0, span = 0;
  for (int64_t x = top; x > 0; --x) {
    // the k items of cost x go to the k least loaded slots, as many at a time as share a load
    for (int64_t k = hist[(size_t)x]; k > 0;) {
      while (load[(size_t)cur] == 0) ++cur;
      const int64_t m = std::min(k, load[(size_t)cur]);
      load[(size_t)cur] -= m;
      load[(size_t)(cur + x)] += m;
      span = std::max(span, cur + x);
      k -= m;
    }
  }
  return span;
}

}  // namespace

pod_attn_status build_plan(const pod_attn_problem& prob, const int32_t* cu, const int32_t* kv,
                           const pod_attn_options& opt, int num_sms, pod_attn_plan_s* plan) {
  const int Hq = prob.num_q_heads, Hkv = prob.num_kv_heads;
  const int Np = prob.num_prefill_seqs, Nd = prob.num_decode_seqs;
  if (Hq < 1 || Hkv < 1 || Np < 0 || Nd < 0 || prob.num_prefill_tokens < 0 ||
      prob.num_blocks < 0 || prob.max_blocks_per_seq < 0 || !std::isfinite(prob.scale) ||
      !(prob.scale > 0.f))
    return POD_ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return POD_ATTN_ERR_INVALID_ARG;
  if (opt.ctas_per_sm < 0 || opt.max_prefill_ctas < 0) return POD_ATTN_ERR_INVALID_ARG;
  // one persistent CTA per SM holds both slots (232 KiB of shared memory, all 512 TMEM columns)
  if (opt.ctas_per_sm > 1) return POD_ATTN_ERR_UNSUPPORTED;
  // head dims 128 and 64 (the layouts are sized for 128; 64 uses their first half)
  if ((prob.head_dim != kHeadDim && prob.head_dim != 64) || prob.block_size != kBlockSize)
    return POD_ATTN_ERR_UNSUPPORTED;
  const int D = prob.head_dim;
  const int G = Hq / Hkv;
  if (G > kMaxGroup) return POD_ATTN_ERR_UNSUPPORTED;
  if ((Np == 0) != (prob.num_prefill_tokens == 0)) return POD_ATTN_ERR_INVALID_ARG;
  if (Np > 0 && cu == nullptr) return POD_ATTN_ERR_INVALID_ARG;
  if (Np + Nd > 0 && (kv == nullptr || prob.num_blocks < 1 || prob.max_blocks_per_seq < 1))
    return POD_ATTN_ERR_INVALID_ARG;
  if (num_sms < 1) return POD_ATTN_ERR_INVALID_ARG;
  // TMA row coordinates of the pools are int32.
  if ((int64_t)prob.num_blocks * Hkv * kBlockSize >= (int64_t(1) << 31))
    return POD_ATTN_ERR_UNSUPPORTED;
  const int64_t max_rows = (int64_t)prob.max_blocks_per_seq * kBlockSize;
  if (Np > 0) {
    if (cu[0] != 0 || cu[Np] != prob.num_prefill_tokens) return POD_ATTN_ERR_INVALID_ARG;
    for (int s = 0; s < Np; ++s) {
      int64_t q = (int64_t)cu[s + 1] - cu[s];
      if (q < 1 || kv[s] < q || kv[s] > max_rows) return POD_ATTN_ERR_INVALID_ARG;
    }
  }
  for (int d = 0; d < Nd; ++d)
    if (kv[Np + d] < 1 || kv[Np + d] > max_rows) return POD_ATTN_ERR_INVALID_ARG;

  plan->prob = prob;
  plan->opt = opt;
  plan->group = G;
  const int hp = G & -G;  // largest power of two dividing G (G <= 8)
  const int tq = kTileM / hp;
  plan->head_pack = hp;
  plan->tile_tokens = tq;
  plan->num_sms = num_sms;
  plan->ctas_per_sm = 1;  // one CTA per SM holds both slots (and all 512 TMEM columns)
  // the cap on CTAs that take prefill items ("POD-Attention" digest, §"가상 CTA와 SM별 균형": the
  // CTAs one prefill may take are limited so decode work is not crowded out); 0 = every CTA
  const int prefill_ctas =
      opt.max_prefill_ctas > 0 ? std::min(opt.max_prefill_ctas, num_sms) : num_sms;
  plan->max_prefill_ctas = prefill_ctas;
  plan->cu.assign(cu ? cu : nullptr, cu ? cu + Np + 1 : nullptr);
  plan->kv.assign(kv ? kv : nullptr, kv ? kv + Np + Nd : nullptr);
  const int64_t slots = (int64_t)num_sms * 2;  // a prefill slot and a decode slot per SM

  // ---- enumerate outputs (before splitting) and their costs --------------------------------
  struct PUnit { int s, t, h; int64_t kend; int64_t ntiles; };
  struct DUnit { int d, g; int64_t L; int64_t nblk; };
  std::vector<PUnit> pu;
  std::vector<DUnit> du;
  int64_t total = 0;
  double pf = 0, pb = 0, db = 0, df = 0;
  const double row_bytes = 4.0 * Hkv * D;  // K + V, bf16
  const bool causal = opt.non_causal == 0;
  for (int s = 0; s < Np; ++s) {
    const int64_t q = (int64_t)cu[s + 1] - cu[s], L = kv[s], P = L - q;
    pf += 4.0 * D * Hq * (double)(causal ? q * P + q * (q + 1) / 2 : q * L);
    pb += (double)L * row_bytes + 4.0 * q * Hq * D;
    for (int64_t t = 0; t < ceil_div(q, (int64_t)tq); ++t) {
      // causal: the tile's last token sees up to its own position; otherwise every row
      const int64_t kend = causal ? P + std::min(q, (t + 1) * tq) : L;
      const int64_t nt = ceil_div(kend, kTileN);
      for (int h0 = 0; h0 < Hq; h0 += hp) {
        pu.push_back({s, (int)t, h0, kend, nt});
        total += nt * kPrefillStepCost;
      }
    }
  }
  for (int d = 0; d < Nd; ++d) {
    const int64_t L = kv[Np + d];
    db += (double)L * row_bytes + 4.0 * Hq * D;
    df += 4.0 * D * Hq * (double)L;
    for (int g = 0; g < Hkv; ++g) {
      du.push_back({d, g, L, ceil_div(L, kBlockSize)});
      total += ceil_div(L, kBlockSize) * kDecodeBlockCost;
    }
  }
  plan->est_prefill_flops = pf;
  plan->est_prefill_bytes = pb;
  plan->est_decode_bytes = db;
  plan->est_decode_flops = df;
  const int64_t target = std::max<int64_t>(1, total / (slots * 4));

  // ---- split and emit ----------------------------------------------------------------------
  // Items are written in enumeration order into flat arrays (cost, 8 words), then ordered
  // longest first; ties keep enumeration order (the sort key carries the item's index).
  struct Split { int64_t ns, chunk; };
  // prefill: one chunk size (steps per item) for all outputs, the one whose items the SMs'
  // prefill slots finish first in the model above; ties keep the larger chunk
  int64_t chunk_p = 0;
  if (!pu.empty() && opt.prefill_splits <= 0) {
    std::vector<int64_t> nts(pu.size()), hist, load;
    int64_t longest = 0;
    for (size_t i = 0; i < pu.size(); ++i) {
      nts[i] = pu[i].ntiles;
      longest = std::max(longest, pu[i].ntiles);
    }
    int64_t best = -1, prev_c = -1;
    for (int k = 1; k <= kMaxPrefillSplits; ++k) {
      const int64_t c = ceil_div(longest, k);
      if (c == prev_c) continue;
      if (k > 1 && c < kMinPrefillTilesPerSplit) break;
      prev_c = c;
      const int64_t t = prefill_makespan(nts, c, prefill_ctas, hist, load);
      if (best < 0 || t < best) {
        best = t;
        chunk_p = c;
      }
    }
  }
  auto split_p = [&](const PUnit& x) {
    int64_t ns;
    if (chunk_p > 0) {
      int64_t chunk;
      rebalanced(x.ntiles, chunk_p, &ns, &chunk);
      return Split{ns, chunk};
    }
    ns = std::max<int64_t>(1, std::min<int64_t>({opt.prefill_splits, x.ntiles,
                                                  (int64_t)kMaxPrefillSplits}));
    const int64_t chunk = ceil_div(x.ntiles, ns);
    return Split{ceil_div(x.ntiles, chunk), chunk};
  };
  // decode-only plans: one chunk size for all outputs, against the groups that run at once
  int64_t chunk_do = 0;
  if (pu.empty() && !du.empty() && opt.decode_splits <= 0) {
    const int64_t groups =
        (int64_t)num_sms * (opt.kv_fp8 ? kDecodeGroupsFp8 : kDecodeGroupsBf16);
    std::vector<int64_t> nblks(du.size());
    int64_t longest = 0;
    for (size_t i = 0; i < du.size(); ++i) {
      nblks[i] = du[i].nblk;
      longest = std::max(longest, du[i].nblk);
    }
    std::vector<int64_t> hist((size_t)(ceil_div(longest, 4) + kDecodeItemOverhead + 1), 0);
    int64_t best = -1, prev_c = -1;
    for (int k : kChunkDivisors) {
      const int64_t c = ceil_div(longest, k);
      if (c == prev_c || (k > 1 && c < kMinDecodeBlocksPerSplit)) continue;
      prev_c = c;
      int64_t n_items = 0;
      for (int64_t n : nblks) {
        int64_t ns, ch;
        rebalanced(n, c, &ns, &ch);
        n_items += ns;
      }
      if (k > 1 && n_items > 4 * groups) break;  // past four waves the tail is already short
      const int64_t t = decode_makespan(nblks, c, groups, hist);
      if (best < 0 || t < best) {  // ties keep the larger chunk (fewer items, fewer merges)
        best = t;
        chunk_do = c;
      }
    }
  }
  auto split_d = [&](const DUnit& x) {
    int64_t ns;
    if (chunk_do > 0) {
      int64_t chunk;
      rebalanced(x.nblk, chunk_do, &ns, &chunk);
      return Split{ns, chunk};
    }
    if (opt.decode_splits > 0) {
      ns = std::min<int64_t>(opt.decode_splits, kMaxDecodeSplits);
    } else {
      ns = ceil_div(x.nblk * kDecodeBlockCost, target);
      ns = std::min<int64_t>(ns, std::max<int64_t>(1, x.nblk / kMinDecodeBlocksPerSplit));
      ns = std::min<int64_t>(ns, kMaxDecodeSplits);
    }
    ns = std::max<int64_t>(1, std::min(ns, x.nblk));
    const int64_t chunk = ceil_div(x.nblk, ns);
    return Split{ceil_div(x.nblk, chunk), chunk};
  };
  std::vector<Split> sp(pu.size()), sd(du.size());
  size_t n_p = 0, n_d = 0, n_units = 0;
  for (size_t i = 0; i < pu.size(); ++i) {
    sp[i] = split_p(pu[i]);
    n_p += (size_t)sp[i].ns;
    n_units += sp[i].ns > 1;
  }
  for (size_t i = 0; i < du.size(); ++i) {
    sd[i] = split_d(du[i]);
    n_d += (size_t)sd[i].ns;
    n_units += sd[i].ns > 1;
  }
  std::vector<int64_t> cost_p(n_p), cost_d(n_d);
  std::vector<int32_t> words_p(n_p * kItemWords), words_d(n_d * kItemWords);
  plan->units.clear();
  plan->units.reserve(n_units * kUnitWords);
  int p_slots = 0, d_slots = 0;
  auto add_unit = [&](int nsplit, int kind) {
    int u = (int)(plan->units.size() / kUnitWords);
    int first = kind == 0 ? p_slots : d_slots;
    (kind == 0 ? p_slots : d_slots) += nsplit;
    plan->units.push_back(nsplit);
    plan->units.push_back(first);
    plan->units.push_back(kind);
    plan->units.push_back(0);
    return u;
  };
  size_t ip = 0, id = 0;
  for (size_t i = 0; i < pu.size(); ++i) {
    const PUnit& x = pu[i];
    const int64_t ns = sp[i].ns, chunk = sp[i].chunk;
    const int u = ns > 1 ? add_unit((int)ns, 0) : -1;
    for (int64_t k = 0; k < ns; ++k, ++ip) {
      const int64_t t0 = k * chunk, t1 = std::min(x.ntiles, (k + 1) * chunk);
      cost_p[ip] = (t1 - t0) * kPrefillStepCost;
      const int32_t w[kItemWords] = {0, x.s, x.t, x.h, (int32_t)(t0 * kTileN),
                                     (int32_t)std::min(x.kend, t1 * kTileN), u, (int32_t)k};
      std::memcpy(&words_p[ip * kItemWords], w, sizeof(w));
    }
  }
  for (size_t i = 0; i < du.size(); ++i) {
    const DUnit& x = du[i];
    const int64_t ns = sd[i].ns, chunk = sd[i].chunk;
    const int u = ns > 1 ? add_unit((int)ns, 1) : -1;
    for (int64_t k = 0; k < ns; ++k, ++id) {
      const int64_t b0 = k * chunk, b1 = std::min(x.nblk, (k + 1) * chunk);
      cost_d[id] = (b1 - b0) * kDecodeBlockCost;
      const int32_t w[kItemWords] = {1, x.d, x.g, 0, (int32_t)(b0 * kBlockSize),
                                     (int32_t)std::min(x.L, b1 * kBlockSize), u, (int32_t)k};
      std::memcpy(&words_d[id * kItemWords], w, sizeof(w));
    }
  }
  // Items are taken longest first. Decode items: by cost, ties in enumeration order (a stable
  // counting sort over the cost in blocks). Prefill items: by cost rounded to a coarse relative
  // bucket (3 significant bits, ~12 % steps), then by split index, then in enumeration order, so
  // that the items running at once share their key ranges (split k of every output reads the
  // same part of its sequence) and keep the K/V rows they read resident in L2, while the order
  // stays longest first to within a bucket.
  auto order = [](const std::vector<int64_t>& key, const std::vector<int32_t>& words,
                  std::vector<int32_t>& out) {  // stable, largest key first
    const size_t n = key.size();
    int64_t top = 0;
    for (int64_t k : key) top = std::max(top, k);
    std::vector<size_t> start((size_t)top + 2, 0);
    for (int64_t k : key) ++start[(size_t)(top - k) + 1];
    for (size_t b = 1; b < start.size(); ++b) start[b] += start[b - 1];
    out.resize(n * kItemWords);
    for (size_t i = 0; i < n; ++i)
      std::memcpy(&out[(start[(size_t)(top - key[i])]++) * kItemWords], &words[i * kItemWords],
                  kItemWords * sizeof(int32_t));
  };
  auto bucket = [](int64_t steps) -> int64_t {  // monotone, 3 significant bits above 15
    if (steps < 16) return steps;
    int bl = 0;
    while ((steps >> bl) != 0) ++bl;
    return 16 + (int64_t)(bl - 5) * 8 + ((steps >> (bl - 4)) & 7);
  };
  for (size_t i = 0; i < n_p; ++i)
    cost_p[i] = bucket(cost_p[i] / kPrefillStepCost) * kMaxPrefillSplits +
                (kMaxPrefillSplits - 1 - words_p[i * kItemWords + 7]);
  for (size_t i = 0; i < n_d; ++i) cost_d[i] /= kDecodeBlockCost;
  order(cost_p, words_p, plan->items_p);
  order(cost_d, words_d, plan->items_d);
  plan->num_p_slots = p_slots;
  // where each token of this iteration sits in its sequence (the KV append writes its K/V
  // row there): chunk token i of prefill sequence s at kv_len - q_len + i, a decode token at
  // kv_len - 1 ("Week 6: Beyond PyTorch: Custom Kernel과 vLLM", §"한 스텝에 여러 종류의 request
  // 섞기": an extend token follows the cached rows, a decode token is the last row)
  plan->new_rows.resize(2 * ((size_t)prob.num_prefill_tokens + Nd));
  size_t r = 0;
  for (int s = 0; s < Np; ++s) {
    const int32_t q = cu[s + 1] - cu[s], P = kv[s] - q;
    for (int32_t i = 0; i < q; ++i, r += 2) {
      plan->new_rows[r] = s;
      plan->new_rows[r + 1] = P + i;
    }
  }
  for (int d = 0; d < Nd; ++d, r += 2) {
    plan->new_rows[r] = Np + d;
    plan->new_rows[r + 1] = kv[Np + d] - 1;
  }
  plan->num_d_slots = d_slots;

  plan->grid_fused = (int)std::min<int64_t>(num_sms, (int64_t)(n_p + n_d));
  plan->grid_prefill = (int)std::min<int64_t>(prefill_ctas, (int64_t)n_p);
  plan->grid_decode = (int)std::min<int64_t>(num_sms, (int64_t)n_d);

  // ---- workspace layout --------------------------------------------------------------------
  WorkspaceLayout& w = plan->ws;
  size_t off = 0;
  w.status = off;
  off += 256;
  w.counters = off;
  w.counter_block_words = kCounterHeader + (size_t)num_sms;
  off = align256(off + kNumModes * w.counter_block_words * 4);
  w.arrive = off;
  off = align256(off + plan->units.size() / kUnitWords * 4);
  w.zero_bytes = off;
  w.items_p = off;
  off = align256(off + plan->items_p.size() * 4);
  w.items_d = off;
  off = align256(off + plan->items_d.size() * 4);
  w.units = off;
  off = align256(off + plan->units.size() * 4);
  w.new_rows = off;
  off = align256(off + plan->new_rows.size() * 4);
  w.partial_p = off;
  off = align256(off + (size_t)p_slots * kPrefillSlotBytes);
  w.partial_d = off;
  off = align256(off + (size_t)d_slots * decode_slot_floats(G) * 4);
  w.records = off;
  if (opt.instrument) off = align256(off + (size_t)(n_p + n_d) * sizeof(pod_attn_item_record));
  w.total = off;

  // the upload image: zeros up to the work lists, then each list at its workspace offset
  std::vector<uint8_t>& img = plan->upload_image;
  img.assign(w.partial_p, 0);
  auto put = [&](size_t at, const std::vector<int32_t>& v) {
    if (!v.empty()) std::memcpy(img.data() + at, v.data(), v.size() * sizeof(int32_t));
  };
  put(w.items_p, plan->items_p);
  put(w.items_d, plan->items_d);
  put(w.units, plan->units);
  put(w.new_rows, plan->new_rows);
  return POD_ATTN_OK;
}

}  // namespace pod
