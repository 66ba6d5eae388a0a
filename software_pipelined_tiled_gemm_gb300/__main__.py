"""Planning reports from the command line (no GPU needed).

    python -m software_pipelined_tiled_gemm_gb300 budget [--m 4096 --n 4096 --k 4096]
        [--dtype f16] [--stages 1 2 3 4 5 6 7 8] [--tile-n N] [--cta-group G]
        [--smem-limit BYTES] [--device INDEX]

For each ring depth, reports the shared memory one CTA needs and what the
planner chooses, marking the depths that do not fit "OVER" (depth 1 is the
single-buffer variant; "6->4" means the planner built fewer slots than
requested because K has only 4 slices).  The TileLang
tutorial's pipelined_gemm.py (chapter 11, "Pipelining and autotuning") has a
report of this kind: its shared_bytes() -- stages x (block_M x block_K +
block_N x block_K) x element size -- checked against a shared-memory limit.
Here the "ring" column is that formula for the tile one CTA holds (with a
CTA pair each CTA holds half of the tile's B rows), and "CTA total" adds
what this kernel needs on top: epilogue staging, barriers and alignment.

The device is the GB300 description (sm_count 152, 227 KiB of shared memory
per block, ...) unless --device queries a GPU; --smem-limit replaces the
shared-memory limit of either.
"""
from __future__ import annotations

import argparse
import sys

from . import (GB300, GEMM_ERR_SMEM_BUDGET, GemmError, describe, gemm_device_query,
               gemm_smem_bytes)


def _device(args) -> dict:
    if args.device is None:
        desc = dict(GB300)
        name = "GB300 description"
    else:
        st, d = gemm_device_query(args.device)
        if st != 0:
            from . import gemm_last_error
            raise SystemExit("gemm_device_query(%d) failed: %s" % (args.device, gemm_last_error()))
        desc = d.as_dict()
        name = "device %d" % args.device
    if args.smem_limit is not None:
        desc["smem_optin"] = int(args.smem_limit)
        name += ", shared-memory limit %d B" % args.smem_limit
    return desc, name


def budget(args, out=sys.stdout) -> int:
    desc, name = _device(args)
    tuning = {}
    if args.tile_n:
        tuning["tile_n"] = args.tile_n
    if args.cta_group:
        tuning["cta_group"] = args.cta_group
    print("%s: %d SMs, %d B shared memory per CTA, L2 %.1f MiB, %d pair clusters"
          % (name, desc["sm_count"], desc["smem_optin"], desc["l2_bytes"] / 2**20,
             desc["pair_clusters"]), file=out)
    print("problem: M=%d N=%d K=%d %s%s" % (args.m, args.n, args.k, args.dtype,
                                            "".join(" %s=%d" % kv for kv in tuning.items())),
          file=out)
    print("%-7s %-12s %-6s %-10s %-10s %-5s %s" % ("stages", "tile", "grid", "ring B",
                                                   "CTA total", "fits", "last wave"), file=out)
    over = 0
    for s in args.stages:
        variant = "single_buffer" if s == 1 else "pipelined"
        try:
            d = describe(args.m, args.n, args.k, args.dtype, stages=s, variant=variant,
                         device=desc, **tuning)
        except GemmError as e:
            if e.status != GEMM_ERR_SMEM_BUDGET:
                raise
            if args.tile_n:            # the requested tile does not fit
                cg = args.cta_group or 1
                tile = "%dx%dx64" % (128 * cg, args.tile_n)
                ring = "%d" % gemm_smem_bytes(128, args.tile_n // cg, 64, 2, s)
            else:                      # no tile width fits
                tile, ring = "none", "-"
            print("%-7d %-12s %-6s %-10s %-10s %-5s %s" % (s, tile, "-", ring, "-", "OVER", "-"),
                  file=out)
            over += 1
            continue
        ring = gemm_smem_bytes(128, d["tile_n"] // d["cta_group"], d["tile_k"], 2, d["stages"])
        if d["stream_k"]:
            wave = "stream-K, %d tiles%s" % (d["tail_tiles"],
                                             " (K halves in clusters)" if d["sk_cluster"] else "")
        elif d["tail_splits"] > 1:
            wave = "%d tiles cut %d ways" % (d["tail_tiles"], d["tail_splits"])
        else:
            wave = "whole tiles"
        depth = "%d" % s if d["stages"] == s else "%d->%d" % (s, d["stages"])
        print("%-7s %-12s %-6d %-10d %-10d %-5s %s" % (
            depth, "%dx%dx%d" % (d["tile_m"], d["tile_n"], d["tile_k"]), d["grid"], ring,
            d["smem_bytes"], "ok", wave), file=out)
    return over


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(prog="python -m software_pipelined_tiled_gemm_gb300")
    sub = ap.add_subparsers(dest="cmd", required=True)
    b = sub.add_parser("budget", help="shared memory and plan per ring depth")
    b.add_argument("--m", type=int, default=4096)
    b.add_argument("--n", type=int, default=4096)
    b.add_argument("--k", type=int, default=4096)
    b.add_argument("--dtype", default="f16", choices=["f16", "bf16"])
    b.add_argument("--stages", type=int, nargs="+", default=list(range(1, 9)))
    b.add_argument("--tile-n", type=int, default=0, choices=[0, 64, 128, 256])
    b.add_argument("--cta-group", type=int, default=0, choices=[0, 1, 2])
    b.add_argument("--smem-limit", type=int, default=None,
                   help="shared memory per CTA in bytes (default: the device's)")
    b.add_argument("--device", type=int, default=None,
                   help="query this CUDA device instead of using the GB300 description")
    args = ap.parse_args(argv)
    if args.cmd == "budget":
        budget(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
