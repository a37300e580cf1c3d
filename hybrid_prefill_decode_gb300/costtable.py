"""Validated latencies of the fused kernel per resource bucket, for an outer scheduler.

The "POD-Attention" digest (Silicon & Systems), §"스케줄링 입력으로 쓰는 자원 특성", argues that
a serving scheduler needs the resource profile of the work, not only token counts, and that the
signal must stay simple enough to use online: describe prefill chunks and decode groups by CTA
count, shared memory, arithmetic intensity and bytes read, in coarse buckets, and let the kernel
publish a few validated (bucket, latency) combinations to choose from. §"예측 가능한 지연시간과
진단" adds that the prefill admitted per iteration should be limited by tail latency, not mean
speed.

Here a batch's bucket is what `pod_attn_plan_bucket` computes in the library (prefill FLOPs and
bytes read, each in power-of-two buckets; CTA counts, shared memory and intensity are reported
alongside). `calibrate` runs the fused kernel through the C ABI on seeded synthetic batches and
records per bucket the p50 and p99 of the measured µs per iteration (cold L2), keeping the worst
figures when several batches fall in one bucket. `lookup` returns the validated entry of a
plan's bucket, or None when that bucket was never measured (outside the validated range: the
caller decides); `choose_chunk` returns the largest candidate prefill chunk whose validated p99
fits a time budget next to a given decode batch.

Command line (on a GPU): python -m hybrid_prefill_decode_gb300.costtable --help
"""
from __future__ import annotations

import argparse
import json
import math
from dataclasses import asdict, dataclass
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

from . import binding as B

Key = Tuple[int, int]


def key_of(bucket: dict) -> Key:
    """The table key of a bucket: (prefill-FLOP bucket, bytes-read bucket)."""
    return (int(bucket["bucket_flops"]), int(bucket["bucket_bytes"]))


@dataclass
class Entry:
    p50_us: float
    p99_us: float
    samples: int          # timed iterations behind the figures
    batches: int          # calibration batches that fell in this bucket
    prefill_ctas: int     # largest CTA counts seen in the bucket
    decode_ctas: int
    intensity: float      # FLOP per byte of the batch that set p99


def _quantile(xs: Sequence[float], q: float) -> float:
    s = sorted(xs)
    return s[min(len(s) - 1, int(round(q * (len(s) - 1))))]


class CostTable:
    """Per-bucket validated latencies of one model shape (q-heads, kv-heads) on one GPU."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, num_sms: int,
                 entries: Optional[Dict[Key, Entry]] = None):
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.num_sms = num_sms
        self.entries: Dict[Key, Entry] = dict(entries or {})

    # ---- building -----------------------------------------------------------------------
    def add(self, bucket: dict, times_us: Sequence[float]) -> None:
        """Record the measured times of one batch; a bucket keeps its worst p50 and p99."""
        if not times_us:
            raise ValueError("no timings")
        k = key_of(bucket)
        p50, p99 = _quantile(times_us, 0.5), _quantile(times_us, 0.99)
        old = self.entries.get(k)
        if old is None:
            self.entries[k] = Entry(p50, p99, len(times_us), 1, int(bucket["prefill_ctas"]),
                                    int(bucket["decode_ctas"]), float(bucket["intensity"]))
            return
        self.entries[k] = Entry(
            max(old.p50_us, p50), max(old.p99_us, p99), old.samples + len(times_us),
            old.batches + 1, max(old.prefill_ctas, int(bucket["prefill_ctas"])),
            max(old.decode_ctas, int(bucket["decode_ctas"])),
            float(bucket["intensity"]) if p99 > old.p99_us else old.intensity)

    # ---- queries ------------------------------------------------------------------------
    def lookup(self, plan: B.Plan) -> Optional[Entry]:
        return self.entries.get(key_of(plan.bucket()))

    def plan_for(self, q_lens: Sequence[int], prefill_kv_lens: Sequence[int],
                 decode_kv_lens: Sequence[int]) -> B.Plan:
        """A host-only plan of a hypothetical batch of this shape (no GPU needed)."""
        cu = [0]
        for q in q_lens:
            cu.append(cu[-1] + q)
        lens = list(prefill_kv_lens) + list(decode_kv_lens)
        maxb = max(1, max((math.ceil(x / 16) for x in lens), default=1))
        nb = max(1, sum(math.ceil(x / 16) for x in lens))
        return B.Plan(self.num_q_heads, self.num_kv_heads, cu if q_lens else [], lens,
                      len(decode_kv_lens), nb, maxb, 1.0 / math.sqrt(128), num_sms=self.num_sms)

    def choose_chunk(self, prefix: int, candidates: Iterable[int],
                     decode_kv_lens: Sequence[int], budget_us: float) -> Optional[int]:
        """The largest chunk c of `candidates` such that one prompt chunk of c tokens after
        `prefix` cached rows, batched with the given decodes, falls in a validated bucket whose
        p99 is within `budget_us`; None if no candidate qualifies."""
        for c in sorted(set(int(x) for x in candidates), reverse=True):
            if c < 1:
                continue
            e = self.lookup(self.plan_for([c], [prefix + c], decode_kv_lens))
            if e is not None and e.p99_us <= budget_us:
                return c
        return None

    # ---- storage ------------------------------------------------------------------------
    def to_json(self) -> str:
        return json.dumps({"num_q_heads": self.num_q_heads, "num_kv_heads": self.num_kv_heads,
                           "num_sms": self.num_sms,
                           "entries": [{"bucket_flops": k[0], "bucket_bytes": k[1], **asdict(e)}
                                       for k, e in sorted(self.entries.items())]}, indent=1)

    @classmethod
    def from_json(cls, text: str) -> "CostTable":
        d = json.loads(text)
        entries = {}
        for e in d["entries"]:
            k = (int(e.pop("bucket_flops")), int(e.pop("bucket_bytes")))
            entries[k] = Entry(**e)
        return cls(d["num_q_heads"], d["num_kv_heads"], d["num_sms"], entries)


def calibrate(num_q_heads: int, num_kv_heads: int, chunks: Sequence[int],
              prefixes: Sequence[int], decode_counts: Sequence[int], decode_ctx: int,
              iters: int = 20, warmup: int = 3, seed: int = 0, device: str = "cuda") -> CostTable:
    """Time the fused kernel on every (chunk, prefix, decode count) combination — seeded
    synthetic batches from the input generator, decode contexts spread over [ctx/2, 3ctx/2) —
    through the C ABI, with the L2 flushed before every timed iteration."""
    import torch
    from . import workloads as W
    dev = torch.device(device)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    table = CostTable(num_q_heads, num_kv_heads, nsm)
    # cold, clean L2 per timed iteration: write 1 GiB, then read 512 MiB (the write's dirty
    # lines are written back here, not inside the timed launch)
    wbuf = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    rbuf = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)
    n = 0
    for c in chunks:
        for pfx in prefixes:
            for nd in decode_counts:
                n += 1
                dl = [max(1, decode_ctx // 2 + (decode_ctx * k) // max(1, nd)) for k in range(nd)]
                q = [c] if c > 0 else []
                b = W.make_batch(num_q_heads, num_kv_heads, q, [pfx + c] if c > 0 else [], dl,
                                 seed=seed + n, device=dev)
                plan = B.Plan.for_batch(b)
                ws = plan.alloc_workspace(dev)
                plan.upload(ws)
                for _ in range(warmup):
                    B.run_batch(plan, b, ws)
                times = []
                for _ in range(iters):
                    wbuf.fill_(1)
                    rbuf.max()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    B.run_batch(plan, b, ws)
                    e1.record()
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1) * 1e3)
                if plan.device_status(ws) != B.OK:
                    raise RuntimeError("device status not OK during calibration")
                table.add(plan.bucket(), times)
                del b, ws
    return table


def main(argv: Optional[List[str]] = None) -> None:
    ap = argparse.ArgumentParser(description="calibrate the fused kernel's per-bucket latencies")
    ap.add_argument("--heads", type=int, nargs=2, default=[32, 8], metavar=("HQ", "HKV"))
    ap.add_argument("--chunks", type=int, nargs="+", default=[256, 512, 1024, 2048])
    ap.add_argument("--prefixes", type=int, nargs="+", default=[4096, 16384])
    ap.add_argument("--decodes", type=int, nargs="+", default=[19, 56])
    ap.add_argument("--decode-ctx", type=int, default=16384)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--out", default=None, help="write the table as JSON here")
    args = ap.parse_args(argv)
    from . import build as build_mod
    build_mod.build()
    t = calibrate(args.heads[0], args.heads[1], args.chunks, args.prefixes, args.decodes,
                  args.decode_ctx, iters=args.iters)
    text = t.to_json()
    if args.out:
        open(args.out, "w").write(text)
    print(text)


if __name__ == "__main__":
    main()
