"""Helpers shared by the GPU tests (inputs from synth, expectations from the oracle)."""
import numpy as np
import torch

import synth
from oracle import lookahead as la
from oracle.model import OracleModel, argmax_lowest


def weights(cfg, seed=0, device="cuda:0"):
    w = synth.llama_weights(cfg, seed, device=device)
    return w


def context(cfg, w, max_ctx, W, N, G):
    from lookahead_decoding_gb300 import lib
    return lib().Context(cfg, w, max_ctx=max_ctx, max_W=W, max_N=N, max_G=G)


def top2_gap(logits):
    s = np.sort(np.asarray(logits, dtype=np.float64))
    return s[-1] - s[-2]
