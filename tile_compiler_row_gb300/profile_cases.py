"""Fixed launch sequences for ncu captures (the commands in ``profiles/``).

Each case builds seeded BF16 inputs of 16384 x 4096 on the GPU (above the L2
with its companions), launches two entry points three times each, in order,
and checks the device status word. An ncu capture picks launches out of
that sequence with ``--launch-skip`` / ``--launch-count``:

    python -m tile_compiler_row_gb300.profile_cases <case>

cases:
  bf16_layernorm  residual LayerNorm, then LayerNorm (seed 3)
  bf16_backward   LayerNorm backward with gamma, then softmax backward (seed 5)
  bwd_gamma       LayerNorm backward with gamma, then without (seed 5)
  affine          affine LayerNorm (gamma, beta), then plain LayerNorm (seed 5)
"""

from __future__ import annotations

import argparse
import sys

ROWS, WIDTH = 16384, 4096


def _rand(gen, *shape):
    import torch
    return torch.rand(*shape, device="cuda", generator=gen)


def run(case: str) -> None:
    import torch

    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    _build.build()
    tile.load()
    torch.cuda.set_device(0)
    bf = torch.bfloat16
    if case == "bf16_layernorm":
        g = torch.Generator(device="cuda").manual_seed(3)
        x = (_rand(g, ROWS, WIDTH) * 2 - 1).to(bf)
        r = (_rand(g, ROWS, WIDTH) * 2 - 1).to(bf)
        y = torch.empty_like(x)
        first = lambda: tile.tile_residual_layernorm_bf16(x, r, y)
        second = lambda: tile.tile_layernorm_bf16(x, y)
    elif case in ("bf16_backward", "bwd_gamma"):
        g = torch.Generator(device="cuda").manual_seed(5)
        x = (_rand(g, ROWS, WIDTH) * 2 - 1).to(bf)
        dy = (_rand(g, ROWS, WIDTH) * 2 - 1).to(bf)
        dx = torch.empty_like(x)
        gam = _rand(g, WIDTH) + 0.5
        first = lambda: tile.tile_layernorm_backward_bf16(x, gam, dy, dx)
        if case == "bf16_backward":
            second = lambda: tile.tile_softmax_backward_bf16(x, dy, dx)
        else:
            second = lambda: tile.tile_layernorm_backward_bf16(x, None, dy, dx)
    elif case == "affine":
        g = torch.Generator(device="cuda").manual_seed(5)
        x = (_rand(g, ROWS, WIDTH) * 2 - 1).to(bf)
        y = torch.empty_like(x)
        gam = _rand(g, WIDTH) + 0.5
        bet = _rand(g, WIDTH) - 0.5
        first = lambda: tile.tile_layernorm_affine_bf16(x, None, gam, bet, y)
        second = lambda: tile.tile_layernorm_bf16(x, y)
    else:
        raise SystemExit(f"unknown case {case!r}")
    for fn in (first, second):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    if tile.tile_check_device_status() != 0:
        raise SystemExit("device status word set")
    print("ok")


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=("bf16_layernorm", "bf16_backward", "bwd_gamma", "affine"))
    run(ap.parse_args(argv).case)
    return 0


if __name__ == "__main__":
    sys.exit(main())
