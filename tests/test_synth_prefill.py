"""The sparse prefill / extend workload: causal, distinct, inside each request's own pages."""
import numpy as np

import synth


def test_prefill_indices_are_causal_distinct_and_inside_the_request():
    B, s_q, prefix, topk = 3, 9, 40, 48
    w = synth.sparse_prefill(seed=5, B=B, s_q=s_q, h_q=64, topk=topk, prefix=prefix)
    assert tuple(w.q.shape) == (B, s_q, 64, 576) and tuple(w.indices.shape) == (B, s_q, topk)
    pages_per_req = (prefix + s_q + synth.PAGE - 1) // synth.PAGE
    idx = w.indices.numpy()
    owner = {}   # page -> request
    for b in range(B):
        for i in range(s_q):
            row = idx[b, i]
            n = min(prefix + i + 1, topk)
            assert (row[:n] >= 0).all() and (row[n:] == -1).all(), (b, i)
            used = row[:n]
            assert len(np.unique(used)) == n
            for page in np.unique(used // synth.PAGE):
                assert owner.setdefault(int(page), b) == b   # no page shared between requests
    # every request uses at most its own number of pages, and a causal row never sees more
    # positions than prefix + i + 1 (token 0 of a prefix of 40 sees 41 positions, 48 slots asked)
    for b in range(B):
        pages = {p for p, r in owner.items() if r == b}
        assert len(pages) <= pages_per_req
    assert (idx[:, 0] == -1).sum(axis=-1).tolist() == [topk - (prefix + 1)] * B
