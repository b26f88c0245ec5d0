"""The sampler's sigma schedule, computed by the library (mmdit_shift_mu,
mmdit_sigma_schedule in include/mmdit.h); this module only marshals it."""
from __future__ import annotations

import ctypes
from typing import List

from . import _lib


def mu_for_tokens(n_img_tokens: int) -> float:
    return float(_lib.load().mmdit_shift_mu(int(n_img_tokens)))


def sigmas(n_steps: int, mu: float) -> List[float]:
    out = (ctypes.c_double * (n_steps + 1))()
    _lib.call("mmdit_sigma_schedule", int(n_steps), float(mu), out)
    return list(out)
