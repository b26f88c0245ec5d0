"""Host-side sigma schedule of the flow-matching sampler.

The pages name an Euler sampler but print no schedule.  Reading taken (the
common shifted-linear choice for Flux-style models): t_i = 1 - i/n for
i = 0..n, sigma_i = s t_i / (1 + (s - 1) t_i) with s = exp(mu), and mu
linear in the image-token count through (256, 0.5) and (4096, 1.15).
The kernels only consume (sigma_i, sigma_{i+1}) pairs.
"""
from __future__ import annotations

import math
from typing import List


def mu_for_tokens(n_img_tokens: int) -> float:
    slope = (1.15 - 0.5) / (4096.0 - 256.0)
    return 0.5 + slope * (n_img_tokens - 256.0)


def sigmas(n_steps: int, mu: float) -> List[float]:
    s = math.exp(mu)
    out = []
    for i in range(n_steps + 1):
        t = 1.0 - i / n_steps
        out.append(s * t / (1.0 + (s - 1.0) * t))
    return out
