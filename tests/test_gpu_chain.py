"""The layer-chain kernel (one launch per stretch between two attention
launches; opt-in with LA_MEGA=1 at la_init) against the multi-launch
schedule of the same call: the same GEMM partition, reduction orders and row
arithmetic, so every needed row's logits must be identical bit for bit,
call after call, and so must the tokens.  la_set_debug bit 4 forces the
multi-launch schedule on a chain context."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import context

pytestmark = pytest.mark.gpu

MID = synth.ModelConfig(n_layers=2, d_model=512, n_heads=4, head_dim=128, d_ffn=1408, vocab=4096, dtype="bf16")
WIDE2 = synth.ModelConfig(n_layers=2, d_model=4096, n_heads=32, head_dim=128, d_ffn=11008, vocab=32000)
FORCE_MULTI = 16


def run_calls(L, ctx, cfg, p, knobs, n_calls, flags):
    L.la_set_debug(ctx.ctx, 1 | flags)
    try:
        out = [L.la_prefill(ctx.ctx, p)]
        logits = []
        for _ in range(n_calls):
            out += L.la_step(ctx.ctx, *knobs)
            lg, need = L.la_debug_logits(ctx.ctx, 1024, cfg.vocab)
            logits.append((need.copy(), lg.copy()))
        return out, logits
    finally:
        L.la_set_debug(ctx.ctx, 0)


@pytest.mark.parametrize("cfg,knobs,plen", [(MID, (15, 5, 15), 96), (MID, (4, 3, 4), 40), (WIDE2, (15, 5, 15), 64)])
def test_chain_equals_multi_launch_bitwise(cfg, knobs, plen, monkeypatch):
    from lookahead_decoding_gb300 import lib
    L = lib()
    w = synth.llama_weights(cfg, 0, device="cuda:0")
    W, N, G = knobs
    monkeypatch.setenv("LA_MEGA", "1")
    ctx = context(cfg, w, max_ctx=512, W=W, N=N, G=G)
    try:
        L.la_set_options(ctx.ctx, L.LA_OPT_POOL_FROM_PROMPT | L.LA_OPT_POOL_FROM_OUTPUT)
        base = synth.markov_zipf_prompt(cfg.vocab, plen // 3, 7).tolist()
        p = (base * 3)[:plen]
        a_out, a_lg = run_calls(L, ctx, cfg, p, knobs, 12, 0)
        b_out, b_lg = run_calls(L, ctx, cfg, p, knobs, 12, FORCE_MULTI)
        assert a_out == b_out
        for (na, la_), (nb, lb) in zip(a_lg, b_lg):
            assert np.array_equal(na, nb)
            assert np.array_equal(la_.view(np.uint32), lb.view(np.uint32))
        # whole requests: lookahead on the chain == AR on the chain == AR multi-launch
        ar = L.la_generate_ar(ctx.ctx, p, 48)
        st_chain = L.la_stats()
        assert L.la_generate(ctx.ctx, p, 48, W, N, G, stats=st_chain) == ar
        L.la_set_debug(ctx.ctx, FORCE_MULTI)
        assert L.la_generate_ar(ctx.ctx, p, 48) == ar
        st_multi = L.la_stats()
        assert L.la_generate(ctx.ctx, p, 48, W, N, G, stats=st_multi) == ar
        L.la_set_debug(ctx.ctx, 0)
        # the chain really ran: fewer kernel launches for the same calls
        assert st_chain.steps == st_multi.steps and st_chain.kernel_launches < st_multi.kernel_launches
    finally:
        ctx.close()
        del w
        torch.cuda.empty_cache()
