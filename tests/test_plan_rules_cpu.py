"""The plan builders' reject rules, on randomly mutated inputs, against a plain restatement.

include/pg.h documents every check pg_plan_paged_prefill, pg_plan_paged_prefill_ring and
pg_plan_paged_segment make before anything is uploaded, and which code wins when several
inputs are wrong (the head relation first, then the sizes, then request by request). This
test restates those rules in Python, draws valid batches, breaks one or two fields at random
and compares the library's status with the restated one. No GPU is involved: every check
runs before the plan touches CUDA, so an input that passes them all returns PG_OK on a GPU
machine and PG_ERR_CUDA here.
"""
import numpy as np
import pytest

from paged_sliding_window_qkv_gb300 import pg

I32 = 2 ** 31 - 1
VALID = "valid"


def restated(kind, a):
    """The status the documented rules give for plan inputs `a` (a dict)."""
    Hq, Hkv, D, ps, R = a["hq"], a["hkv"], a["d"], a["ps"], a["num_req"]
    if Hkv == 0:
        return pg.PG_ERR_ZERO_KV_HEADS
    if Hkv < 0 or Hq <= 0 or Hq % Hkv != 0:
        return pg.PG_ERR_HEADS
    if D <= 0 or D % 2 != 0 or ps <= 0:
        return pg.PG_ERR_ARG
    qo, kvp, start = a["qo"], a["kvp"], a["start"]
    if R > 0 and (qo[0] != 0 or kvp[0] != 0):
        return pg.PG_ERR_ARG
    for r in range(R):
        q0, q1, k0, k1 = int(qo[r]), int(qo[r + 1]), int(kvp[r]), int(kvp[r + 1])
        if q1 <= q0 or k1 <= k0:
            return pg.PG_ERR_ARG
        if q1 > I32 or k1 > I32:
            return pg.PG_ERR_I32_OVERFLOW
        sp = int(start[r])
        if sp < 0:
            return pg.PG_ERR_ARG
        pos_end = sp + q1 - q0
        if pos_end > I32:
            return pg.PG_ERR_I32_OVERFLOW
        if kind == "ring":
            cap, need = (k1 - k0) * ps, a["window"] + q1 - q0
            if cap < need and pos_end > cap:
                return pg.PG_ERR_COVERAGE
            continue
        lpl = int(a["last"][r])
        if lpl < 1 or lpl > ps:
            return pg.PG_ERR_LAST_PAGE_LEN
        kv = (k1 - k0 - 1) * ps + lpl
        if kind == "segment":
            s0 = int(a["kv_start"][r])
            if s0 < 0:
                return pg.PG_ERR_ARG
            kv += s0
        if kv > I32:
            return pg.PG_ERR_I32_OVERFLOW
        if kind == "linear" and kv != pos_end:
            return pg.PG_ERR_COVERAGE
        if kind == "segment" and kv > pos_end:
            return pg.PG_ERR_COVERAGE
    npages = int(kvp[R]) if R > 0 else 0
    if (np.asarray(a["pages"][:npages]) < 0).any():
        return pg.PG_ERR_PAGE_OOB
    return VALID


def call(kind, a):
    common = (None, a["num_req"], a["qo"], a["kvp"], a["pages"])
    geo = (a["hq"], a["hkv"], a["d"], a["ps"])
    if kind == "linear":
        return pg.pg_plan_paged_prefill(*common, a["last"], a["start"], *geo, stream=0)[0]
    if kind == "ring":
        return pg.pg_plan_paged_prefill_ring(*common, a["start"], *geo, a["window"], stream=0)[0]
    return pg.pg_plan_paged_segment(*common, a["last"], a["kv_start"], a["start"], *geo,
                                    stream=0)[0]


def valid_inputs(rng, kind):
    R = int(rng.integers(1, 5))
    ps = int(rng.choice([4, 8, 16]))
    qo_lens = rng.integers(1, 40, R)
    start = rng.integers(0, 200, R)
    window = int(rng.integers(0, 64))
    if kind == "ring":
        need = window + qo_lens
        npages = -(-need // ps) + rng.integers(0, 3, R)
        last = np.ones(R, np.int32)
        kv_start = np.zeros(R, np.int64)
    else:
        kv_start = rng.integers(0, 50, R) if kind == "segment" else np.zeros(R, np.int64)
        if kind == "segment":
            kv_start = np.minimum(kv_start, start + qo_lens - 1)
        n = start + qo_lens - kv_start             # keys held, ending at the step's end
        npages = -(-n // ps)
        last = (n - (npages - 1) * ps).astype(np.int32)
    qo = np.zeros(R + 1, np.int64)
    qo[1:] = np.cumsum(qo_lens)
    kvp = np.zeros(R + 1, np.int64)
    kvp[1:] = np.cumsum(npages)
    pages = rng.permutation(int(kvp[-1]) + 8)[: int(kvp[-1])].astype(np.int32)
    hkv = int(rng.choice([1, 2, 8]))
    return dict(num_req=R, qo=qo, kvp=kvp, pages=pages, last=last, start=start.astype(np.int64),
                kv_start=kv_start.astype(np.int64), window=window, hq=hkv * int(rng.choice([1, 2, 8])),
                hkv=hkv, d=int(rng.choice([256, 512])), ps=ps)


MUTATIONS = [
    lambda a, r: a.update(hkv=0),
    lambda a, r: a.update(hkv=-a["hkv"]),
    lambda a, r: a.update(hq=a["hkv"] * 3 + 1 if a["hkv"] > 1 else 0),
    lambda a, r: a.update(d=a["d"] + 1),
    lambda a, r: a.update(ps=0),
    lambda a, r: a["qo"].__setitem__(0, 1),
    lambda a, r: a["kvp"].__setitem__(0, 1),
    lambda a, r: a["qo"].__setitem__(-1, a["qo"][-2]),             # an empty request
    lambda a, r: a["kvp"].__setitem__(-1, a["kvp"][-2]),           # a request with no pages
    lambda a, r: a["start"].__setitem__(int(r.integers(a["num_req"])), -1),
    lambda a, r: a["start"].__setitem__(int(r.integers(a["num_req"])), I32),  # past int32
    lambda a, r: a["last"].__setitem__(int(r.integers(a["num_req"])), 0),
    lambda a, r: a["last"].__setitem__(int(r.integers(a["num_req"])), a["ps"] + 1),
    lambda a, r: a["start"].__setitem__(int(r.integers(a["num_req"])),
                                        a["start"][0] + int(r.choice([-1, 1]))),  # coverage
    lambda a, r: a["pages"].__setitem__(int(r.integers(max(1, len(a["pages"])))), -3),
    lambda a, r: a["kv_start"].__setitem__(int(r.integers(a["num_req"])), -1),
    lambda a, r: a["kv_start"].__setitem__(int(r.integers(a["num_req"])), 10 ** 6),
    lambda a, r: a.update(window=a["window"] + int(r.integers(1, 200))),   # ring too short
]


@pytest.mark.parametrize("kind", ["linear", "ring", "segment"])
def test_random_plan_inputs_follow_the_documented_rules(kind):
    rng = np.random.Generator(np.random.PCG64({"linear": 1, "ring": 2, "segment": 3}[kind]))
    seen = set()
    for case in range(600):
        a = valid_inputs(rng, kind)
        for _ in range(int(rng.integers(0, 3))):       # zero, one or two broken fields
            MUTATIONS[int(rng.integers(len(MUTATIONS)))](a, rng)
        want = restated(kind, a)
        got = call(kind, a)
        if want == VALID:
            assert got in (pg.PG_OK, pg.PG_ERR_CUDA), (case, kind, got)
        else:
            assert got == want, (case, kind, pg.pg_status_string(got), pg.pg_status_string(want))
        seen.add(want)
    assert VALID in seen and len(seen) >= 5          # both valid and several reject kinds drawn
