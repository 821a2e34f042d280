"""The GPU tests' error metrics, checked on the CPU with planted errors: the per-tile bar
catches one wrong row of one head that the whole-tensor rel-RMS lets through, and the
whole-tensor metrics see what they should."""
import numpy as np
import torch

from tests import gpu_util as gu


def _pair(seed=0, shape=(2, 3, 512, 64)):
    rng = np.random.default_rng(seed)
    ref = {n: rng.standard_normal(shape) for n in ("dq", "dk", "dv")}
    ref["o"] = rng.standard_normal(shape)
    ref["lse"] = rng.standard_normal(shape[:3])
    # the kernel's outputs: the reference rounded to bf16 (relative error up to 2^-9)
    gpu = {n: torch.from_numpy(r).to(torch.bfloat16) for n, r in ref.items() if n != "lse"}
    gpu["lse"] = torch.from_numpy(ref["lse"]).float()
    return gpu, ref


def test_rounding_alone_passes_every_bar():
    gpu, ref = _pair()
    gu.assert_within_tolerance(gu.compare(gpu, ref))
    gu.assert_tiles_within_tolerance(gu.tile_errors(gpu, ref))


def test_one_wrong_row_fails_the_tile_bar_only():
    gpu, ref = _pair(1, (4, 16, 512, 32))
    bad = gpu["dk"].clone()
    bad[1, 2, 300] = 0  # one row of one head lost
    gpu["dk"] = bad
    err = gu.compare(gpu, ref)
    assert err["dk"][1] <= gu.TOL_GRAD_REL_RMS  # hidden in the whole tensor ...
    terr = gu.tile_errors(gpu, ref)
    assert terr["dk"][1] == (1, 2, 256)          # ... but not in its tile
    assert terr["dk"][0] > gu.TOL_GRAD_TILE_REL_RMS
    assert terr["dq"][0] <= gu.TOL_GRAD_TILE_REL_RMS


def test_every_helper_the_tests_use_exists():
    import glob
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    used = set()
    for f in glob.glob(os.path.join(root, "tests", "*.py")) + [os.path.join(root, "__graft_entry__.py")]:
        used |= set(re.findall(r"\bgu\.(\w+)", open(f).read()))
    assert not [n for n in sorted(used) if not hasattr(gu, n)]
