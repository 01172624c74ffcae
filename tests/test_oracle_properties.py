"""Property test of the oracle's three forms on random tiny problems: the
recurrence, the dense semiseparable matrix and the block decomposition must
agree for any shape, packing, chunk size and optional inputs."""
import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle


@st.composite
def problems(draw):
    G = draw(st.integers(1, 3))
    H = G * draw(st.integers(1, 2))
    P = draw(st.integers(1, 3))
    N = draw(st.integers(1, 4))
    packed = draw(st.booleans())
    if packed:
        lens = draw(st.lists(st.integers(0, 6), min_size=1, max_size=4))
        b, L = 1, sum(lens)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        nseq = len(lens)
    else:
        b, L, cu = draw(st.integers(1, 2)), draw(st.integers(1, 12)), None
        nseq = b
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.standard_normal((b, L, H, P)),
        dt=rng.uniform(0.0, 1.0, (b, L, H)),
        A=-rng.uniform(0.0, 4.0, H),
        B=rng.standard_normal((b, L, G, N)),
        C=rng.standard_normal((b, L, G, N)),
        D=rng.standard_normal(H) if draw(st.booleans()) else None,
        initial_states=rng.standard_normal((nseq, H, P, N)) if draw(st.booleans()) else None,
        cu_seqlens=cu,
    ), draw(st.integers(1, 7))


def _close(a, b):
    scale = max(np.abs(b).max(), 1.0) if b.size else 1.0
    return np.abs(a - b).max() <= 1e-10 * scale if b.size else True


@settings(max_examples=150, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(problems())
def test_three_forms_agree(case):
    args, chunk = case
    yr, fr = oracle.recurrent(**args)
    yq, fq = oracle.quadratic(**args)
    yc, fc = oracle.chunked(chunk=chunk, **args)
    assert _close(yq, yr) and _close(fq, fr)
    assert _close(yc, yr) and _close(fc, fr)
