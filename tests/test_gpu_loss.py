"""GPU parity of the loss-boundary kernels (include/tree_loss.h) against the
oracle: weights folded into rows (bit-exact against an fp32 product rounded to
bf16), per-trajectory log-probs (|err| <= 2e-4 against fp64: fp32 sums over
the vocabulary) and subtree advantages (|err| <= 1e-4 against fp64)."""
import numpy as np
import pytest
import torch

from oracle import layout as OL
from oracle import loss as OLS
from prefix_tree_attention_attn_gb300 import TreePlan, device_status
from prefix_tree_attention_attn_gb300 import loss as TL
from workloads import trees as WT

pytestmark = pytest.mark.gpu

LP_TOL = 2e-4
ADV_TOL = 1e-4


@pytest.fixture(autouse=True)
def _lib(lib, cuda_device):
    yield
    torch.cuda.synchronize()
    assert device_status() == 0


def test_scale_rows_bit_exact():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(1001, 32, 128, generator=g).to(torch.bfloat16)
    w = (torch.rand(1001, generator=g) * 4).float()
    w[::7] = 1.0
    y = TL.scale_rows(x.cuda(), w.cuda()).cpu()
    want = (x.float() * w[:, None, None]).to(torch.bfloat16)
    assert torch.equal(y, want)
    z = x.cuda().clone()
    TL.scale_rows(z, w.cuda(), out=z)                 # in place
    assert torch.equal(z.cpu(), want)


def draw_logits(N, V, seed):
    g = torch.Generator().manual_seed(seed)
    logits = (torch.randn(N, V, generator=g) * 2.0).to(torch.bfloat16)
    tokens = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    return logits, tokens


@pytest.mark.parametrize("name,V", [("tiny_binary", 1000), ("segment_tree", 4096), ("grpo_star", 2048)])
def test_traj_logprobs_full(name, V):
    t = WT.load_tree(name)
    plan = TreePlan(t.parent, t.seg_len)
    logits, tokens = draw_logits(t.n_tokens, V, 7)
    lse, lp = TL.traj_logprobs(plan, logits.cuda(), tokens.cuda())
    x = logits.double().numpy()
    rl = OLS.row_logsumexp(x)
    assert np.abs(lse.cpu().double().numpy() - rl).max() <= LP_TOL
    want = OLS.traj_logprobs(t.parent, t.seg_len, x, tokens.numpy(), rows_lse=rl)
    assert lp.shape[0] == want.shape[0] == t.n_expanded - len(OL.leaves(t.parent))
    assert np.abs(lp.cpu().double().numpy() - want).max() <= LP_TOL


def test_traj_logprobs_qwen_vocab_sampled():
    # the LM-head width of the Qwen2.5 models the TreePO page trains (152,064)
    t = WT.load_tree("grpo_star")
    plan = TreePlan(t.parent, t.seg_len)
    V = 152064
    g = torch.Generator(device="cuda").manual_seed(9)
    logits = (torch.randn(t.n_tokens, V, generator=g, device="cuda") * 2.0).to(torch.bfloat16)
    tokens = torch.randint(0, V, (t.n_tokens,), generator=g, device="cuda", dtype=torch.int32)
    lse, lp = TL.traj_logprobs(plan, logits, tokens)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(t.n_tokens, size=64, replace=False)
    sub = logits[torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
    rl = OLS.row_logsumexp(sub)
    assert np.abs(lse.cpu().double().numpy()[rows] - rl).max() <= LP_TOL
    # predictions made from the sampled rows
    _, ptr, tok = TL.trajectories(plan)
    tk = tokens.cpu().numpy()
    lpc = lp.cpu().double().numpy()
    where = {int(r): i for i, r in enumerate(rows)}
    k = 0
    checked = 0
    for l in range(len(ptr) - 1):
        for p in range(ptr[l], ptr[l + 1] - 1):
            r, s = int(tok[p]), int(tok[p + 1])
            if r in where:
                want = sub[where[r], tk[s]] - rl[where[r]]
                assert abs(lpc[k] - want) <= LP_TOL
                checked += 1
            k += 1
    assert checked > 0 and k == lp.shape[0]


def test_traj_logprobs_bad_token_is_nan():
    t = WT.Tree("s", [-1, 0], [3, 2])
    plan = TreePlan(t.parent, t.seg_len)
    logits, tokens = draw_logits(5, 64, 1)
    tokens[4] = 64                                     # out of range: predicted from row 3
    _, lp = TL.traj_logprobs(plan, logits.cuda(), tokens.cuda())
    v = lp.cpu().numpy()
    assert np.isnan(v[3]) and np.isfinite(v[:3]).all()


FLAGS = [0, TL.NORM_STD, TL.SIZE_WEIGHTED, TL.NO_ROOT, TL.NORM_STD | TL.SIZE_WEIGHTED | TL.NO_ROOT]


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("name", ["tiny_binary", "segment_tree", "agentic_tree", "random"])
def test_subtree_advantage(name, flags):
    if name == "random":
        t = WT.random_tree(np.random.default_rng(4), 40, [1, 2, 9], n_roots=3)
    else:
        t = WT.load_tree(name)
    plan = TreePlan(t.parent, t.seg_len)
    L = len(OL.leaves(t.parent))
    r = torch.tensor(np.random.default_rng(flags).normal(size=L), dtype=torch.float32)
    adv, nc, tc = TL.subtree_advantage(plan, r.cuda(), flags=flags, eps=1e-4)
    A, NC, TC = OLS.subtree_advantage(t.parent, t.seg_len, r.double().numpy(), norm_std=bool(flags & 1),
                                      size_weighted=bool(flags & 2), no_root=bool(flags & 4), eps=1e-4)
    assert np.abs(adv.cpu().double().numpy() - A).max() <= ADV_TOL
    assert np.abs(nc.cpu().double().numpy() - NC).max() <= ADV_TOL * max(1, L / 16)
    assert np.abs(tc.cpu().double().numpy() - TC).max() <= ADV_TOL * max(1, L / 16)
