"""The journal's dependency-chain summary (profile_step.chain) on a synthetic journal whose
answer is fixed by construction: two CTAs, three layers, every op a fixed time after the
previous one."""
from persistent_sm_decode_megakernel_gb300.profile_step import chain


def _journal():
    recs = []
    t = 0
    # per op: (stage delay after the previous op's last end, work after staging) in ns
    plan = {2: (1500, 3000), 3: (500, 2000), 4: (None, 1500), 5: (300, 2500), 6: (1200, 9000), 7: (600, 4000)}
    for layer in range(3):
        for op in (2, 3, 4, 5, 6, 7):
            stage, work = plan[op]
            ends = []
            for cta, skew in ((0, 0), (1, 200)):
                fetch = t
                m0 = t + stage + skew if stage is not None else 0
                end = (m0 if stage is not None else t + skew) + work
                recs.append((cta, 0, op, layer, fetch, fetch, end, m0, 0, 0, 0, 0, 0))
                ends.append(end)
            t = max(ends)
    return recs


def test_chain_reports_staging_ends_and_hops():
    c = chain(_journal())
    # layer boundaries are the previous layer's last down end; the QKV hop is its stage delay
    assert c["qkv"]["hop"] == 1.5
    assert c["qkv"]["staged"] == 1.6          # median of 1.5 and 1.7
    assert c["attn"]["hop"] == 0.5
    assert "staged" not in c["reduce"] and "hop" not in c["reduce"]
    assert c["oproj"]["hop"] == 0.3
    assert c["upgate"]["hop"] == 1.2
    assert c["down"]["hop"] == 0.6
    # the down projection ends a whole layer after the reference: the sum of the chain
    layer_us = (1.5 + 0.2 + 3.0) + (0.5 + 0.2 + 2.0) + (0.2 + 1.5) + (0.3 + 0.2 + 2.5) + (1.2 + 0.2 + 9.0) + (0.6 + 0.2 + 4.0)
    assert abs(c["down"]["end_max"] - layer_us) < 1e-6
