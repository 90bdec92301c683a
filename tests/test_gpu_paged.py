"""The paged KV cache (hy_cache_alloc_paged: one pool of 128-token pages,
a page table per sequence) through the C ABI: against the FP64 oracle,
against the contiguous cache, and under continuous batching (sequences
joining and leaving a batch between steps, their pages reused), with the pool
accounting and its capacity refusal.  Tolerances as in the decode tests."""
import numpy as np
import pytest

from bandwidth_bound_hybrid_gb300 import capi
from oracle import oracle as orc
from synth import workloads
from tests.gpu_util import rel_l2, to_np

pytestmark = pytest.mark.gpu

LOGIT_TOL, HIDDEN_TOL, ID_MARGIN = 1e-2, 5e-3, 0.05
SHAPE = workloads.TINY


@pytest.fixture(scope="module")
def W(gpu):
    from bandwidth_bound_hybrid_gb300 import build
    build.build()
    return workloads.device_weights(SHAPE), workloads.host_weights(SHAPE)


def _t(x):
    import torch
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def check(got, r, what):
    e = rel_l2(got, r["logits"])
    assert e <= LOGIT_TOL, f"{what}: logits rel-L2 {e:.3g}"
    return e


def test_paged_cache_against_the_oracle(W):
    """A 150-token prompt (two pages, the second partly filled) through the
    chunked prefill, then 10 decode steps, per-layer hidden states too."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    dev_w, host_w = W
    model = HybridModel(SHAPE, dev_w, [300], flags=capi.HY_FLAG_DEBUG, pages=(128, 4))
    ref = orc.Oracle(SHAPE, host_w, 300)
    prompt = workloads.host.uniform_ids(4, workloads.PROMPT_TID, 150, SHAPE.vocab)
    lg = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
    model.prefill(0, torch.from_numpy(prompt).cuda(), lg)
    assert model.free_pages() == 2
    for t in prompt:
        r = ref.forward(int(t))
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    for s in range(10):
        torch.cuda.synchronize()
        check(to_np(lg), r, f"step {s}")
        for l in range(SHAPE.n_layers):
            assert rel_l2(to_np(model.debug_hidden(l)), r["hidden"][l]) <= HIDDEN_TOL
        nxt = int(orc.argmax(r["logits"]))
        model.decode_step(0, _t([nxt]), ids, lg)
        r = ref.forward(nxt)
    assert model.check_device() == 0
    model.close()


def test_paged_equals_contiguous(W):
    """The same prompt and steps on a paged and a contiguous cache: the
    paged cache splits the KV scan at tile boundaries (another order of the
    same sums), so the logits agree to rounding and the greedy ids match."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    dev_w, _ = W
    prompt = workloads.host.uniform_ids(6, workloads.PROMPT_TID, 260, SHAPE.vocab)
    outs = []
    for pages in (None, (128, 3)):
        m = HybridModel(SHAPE, dev_w, [300], pages=pages)
        lg = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        m.prefill(0, torch.from_numpy(prompt).cuda(), lg)
        seq = []
        tok = _t([11])
        for _ in range(8):
            m.decode_step(0, tok, ids, lg)
            torch.cuda.synchronize()
            seq.append((int(ids.item()), to_np(lg).copy()))
            tok = ids.clone()
        assert m.check_device() == 0
        m.close()
        outs.append(seq)
    for (a, la), (b, lb) in zip(*outs):
        assert a == b
        assert rel_l2(lb, la) < 1e-5


def test_synthetic_fill_through_pages_equals_contiguous(W):
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    dev_w, _ = W
    got = []
    for pages in (None, (128, 4)):
        m = HybridModel(SHAPE, dev_w, [400], pages=pages)
        m.fill_synthetic(0, 333, seed=9)
        lg = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        m.decode_step(0, _t([5]), ids, lg)
        torch.cuda.synchronize()
        got.append(to_np(lg).copy())
        if pages:
            assert m.free_pages() == 1
        m.close()
    assert rel_l2(got[1], got[0]) < 1e-5


def test_continuous_batching_over_a_shared_pool(W):
    """Four sequence slots of capacity 512 share a pool of 6 pages (768
    positions).  Sequences join (prefill) and leave (reset) between batched
    steps; a leaving sequence's pages serve the next one; every live
    sequence is checked against its own oracle at every step; a prefill the
    pool cannot hold is refused with nothing taken."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    dev_w, host_w = W
    model = HybridModel(SHAPE, dev_w, [512] * 4, pages=(128, 6))
    refs, last = {}, {}

    def join(s, n):
        prompt = workloads.host.uniform_ids(20 + s, workloads.PROMPT_TID, n, SHAPE.vocab)
        lg = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
        model.prefill(s, torch.from_numpy(prompt).cuda(), lg)
        refs[s] = orc.Oracle(SHAPE, host_w, 512)
        for t in prompt:
            r = refs[s].forward(int(t))
        torch.cuda.synchronize()
        check(to_np(lg), r, f"sequence {s} after its prompt")
        last[s] = r

    def steps(live, n):
        lg = torch.empty((len(live), SHAPE.vocab), dtype=torch.float32, device="cuda")
        ids = torch.empty(len(live), dtype=torch.int32, device="cuda")
        for k in range(n):
            toks = [int(orc.argmax(last[s]["logits"])) for s in live]
            model.decode_batch(live, _t(toks), ids, lg)
            torch.cuda.synchronize()
            got = to_np(lg)
            for i, (s, t) in enumerate(zip(live, toks)):
                last[s] = refs[s].forward(t)
                check(got[i], last[s], f"step {k} of batch {live}, sequence {s}")
                srt = np.sort(last[s]["logits"])
                if srt[-1] - srt[-2] > ID_MARGIN:
                    assert int(ids[i].item()) == int(orc.argmax(last[s]["logits"]))

    join(0, 100)
    join(1, 130)
    assert model.free_pages() == 3
    steps([0, 1], 5)
    join(2, 60)
    assert model.free_pages() == 2
    steps([0, 1, 2], 5)
    # a 400-token prompt needs 4 pages: refused, nothing taken, nothing launched
    with pytest.raises(capi.HybridError) as ei:
        model.prefill(3, torch.zeros(400, dtype=torch.int32, device="cuda"))
    assert ei.value.code == capi.HY_ERR_CAPACITY
    assert model.free_pages() == 2 and model.seq_len(3) == 0
    model.reset(0)  # sequence 0 leaves: its page returns to the pool
    del refs[0], last[0]
    assert model.free_pages() == 3
    join(3, 200)  # two pages, one of them sequence 0's
    assert model.free_pages() == 1
    steps([1, 2, 3], 5)
    assert model.check_device() == 0
    model.close()


def test_long_context_paged_equals_contiguous(gpu):
    """Four layers of the dense 4B shape from a 16384-token synthetic context
    on a paged and on a contiguous cache: the long-context split count runs
    the attention as CTA pairs, on both layouts; the logits agree to
    rounding (the paged scan splits at tile boundaries)."""
    import dataclasses

    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l4-long", n_layers=4, attn_layers=(3,))
    dev_w = workloads.device_weights(shape)
    cap, ctx = 16384 + 128, 16384
    got = []
    for pages in (None, (128, cap // 128)):
        m = HybridModel(shape, dev_w, [cap], pages=pages)
        m.fill_synthetic(0, ctx, seed=3)
        lg = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        tok = _t([7])
        seq = []
        for _ in range(3):
            m.decode_step(0, tok, ids, lg)
            torch.cuda.synchronize()
            seq.append((int(ids.item()), to_np(lg).copy()))
            tok = ids.clone()
        assert m.check_device() == 0
        m.close()
        got.append(seq)
    del dev_w
    for (a, la), (b, lb) in zip(*got):
        assert a == b
        assert rel_l2(lb, la) < 1e-5
