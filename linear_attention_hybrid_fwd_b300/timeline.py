"""Per-stage timeline of the tensor-core prefill on the 8K-token workload.

``python -m linear_attention_hybrid_fwd_b300.timeline [--activated]`` builds the library
with ``-DLA_TIMELINE`` (``liblightning_attn_timeline.so``), runs the B1 H64 N8192 prefill,
reads back the ``%globaltimer`` stamps that every CTA wrote for its first 64 chunks, and
prints the median time of each stage over chunks 10..55 of the 128 head CTAs.  The
stamps cost time of their own (the instrumented kernel runs about 10% slower), so the
table explains where a chunk's time goes; the kernel's speed comes from bench.py.

Event numbers (per CTA and chunk):
  0 q or k load issued        1 v load issued            2 g load issued
  3 SiLU: raw tile landed     4 SiLU: own tile done      5 SiLU: raw v landed
  6 SiLU: all done            7 MMA: own and peer tiles  27 MMA: score buffer free
  8 MMA: scores issued        28 MMA: y buffer free      29 MMA: bf16 state ready
  9 MMA: Q^S, K^T V issued    30/31 MMA: P half 0/1 seen 10 MMA: P V issued
  11 conversion: state done   12 conversion: bf16 state  13/15 mask: score half seen
  14/16 mask: P half written  17 post: y ready           18 post: partials counted
  19/22 finish 0/1: norm factor   20/23 finish 0/1: y and g ready
  21/24 finish 0/1: out tile written
  25 reducer: chunk complete  26 reducer: factors published
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

CTAS, CHUNKS, EVENTS = 160, 64, 32
C0, C1 = 10, 56  # steady-state chunks

STAGES = [
    ("chunk period (MMA warp, chunk to chunk)", 7, 7, 1),
    ("q/k load issue -> landed", 3, 0, 0),
    ("SiLU of the own 128x128 tile", 4, 3, 0),
    ("SiLU of this CTA's 128x64 v", 6, 5, 0),
    ("own SiLU done -> peer tile seen (DSMEM push)", 7, 6, 0),
    ("MMA: score buffer free -> 8 score MMAs issued", 8, 27, 0),
    ("MMA: bf16 state ready -> 16 Q^S, K^T V MMAs issued", 9, 29, 0),
    ("MMA: P half 1 seen -> P V issued (4 MMAs, commits)", 10, 31, 0),
    ("conversion: fp32 state -> bf16 operand", 12, 11, 0),
    ("mask: score half 0 -> P half 0", 14, 13, 0),
    ("mask: P half 0 -> P half 1", 16, 14, 0),
    ("post: y ready -> partials counted", 18, 17, 0),
    ("finish: y and g ready -> out tile written", 21, 20, 0),
    ("post -> norm factor seen (cross-head exchange)", 19, 18, 0),
]


def analyse(stamps: np.ndarray) -> list[tuple[str, float, float, float]]:
    heads = stamps[:128].astype(np.int64)
    t0 = heads[heads > 0].min()
    rel = np.where(heads > 0, heads - t0, -(10 ** 12)) / 1000.0  # us
    rows = []
    for name, e1, e0, lag in STAGES:
        x = (rel[:, C0 + lag:C1 + lag, e1] - rel[:, C0:C1, e0]).ravel()
        x = x[np.abs(x) < 1e5]
        rows.append((name, float(np.median(x)), float(np.percentile(x, 10)),
                     float(np.percentile(x, 90))))
    return rows


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    activated = "--activated" in argv
    import torch
    from . import build as la_build
    import linear_attention_hybrid_fwd_b300 as la
    from .inputs import make_prefill_inputs
    la._LIB_PATH = la_build.build_timeline()
    lib = la.load_library()
    lib.la_timeline_fetch.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    dev = torch.device("cuda", 0)
    q, k, v, g = make_prefill_inputs(1, 8192, 64, 128, torch.bfloat16, 0.5, 2, dev)
    out = torch.empty_like(q)
    S = torch.empty((1, 64, 128, 128), device=dev, dtype=torch.float32)
    for _ in range(3):
        la.la_prefill(q, k, v, g, out=out, kv_state_out=S, activated=activated)
    torch.cuda.synchronize()
    assert lib.la_timeline_clear() == 0
    la.la_prefill(q, k, v, g, out=out, kv_state_out=S, activated=activated)
    torch.cuda.synchronize()
    if la.la_get_device_status() != 0:
        raise SystemExit("device status error")
    buf = np.zeros(CTAS * CHUNKS * EVENTS, dtype=np.uint64)
    assert lib.la_timeline_fetch(buf.ctypes.data, buf.nbytes) == 0
    rows = analyse(buf.reshape(CTAS, CHUNKS, EVENTS))
    print(f"k_prefill_tc timeline, B1 H64 N8192, {'activated' if activated else 'raw'} "
          f"inputs, chunks {C0}..{C1 - 1} of 128 head CTAs (us)")
    print(f"{'stage':52s} {'median':>7s} {'p10':>7s} {'p90':>7s}")
    for name, med, p10, p90 in rows:
        print(f"{name:52s} {med:7.2f} {p10:7.2f} {p90:7.2f}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
