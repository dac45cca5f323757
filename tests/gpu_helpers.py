"""Helpers for the GPU parity tests: product objects built through the C ABI,
oracle objects built by the oracle, and the same seeded inputs for both."""

import functools

import numpy as np

from oracle.step import pack_bitmask
from tests.oracle_cache import oracle_dfa, vocab
from workloads import GRAMMARS, make_logits


@functools.lru_cache(maxsize=None)
def product_grammar(name: str):
    from grammar_constrained_decoding_gb300 import Bounds, Grammar
    spec = GRAMMARS[name]
    b = spec.bounds
    return Grammar.compile(spec.source, spec.kind,
                           Bounds(b.ws_max, b.max_len_default, b.depth_max, b.max_items_default, b.max_tokens))


@functools.lru_cache(maxsize=None)
def product_vocab(kind: str, V: int):
    from grammar_constrained_decoding_gb300 import Vocab
    return Vocab(vocab(kind, V))


def make_ctx(names, kind, V):
    from grammar_constrained_decoding_gb300 import Ctx
    return Ctx([product_grammar(n) for n in names], product_vocab(kind, V))


def dev(x, dtype=None):
    import torch
    t = torch.as_tensor(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def empty(shape, dtype):
    import torch
    return torch.empty(shape, dtype=dtype, device="cuda")


def host(t) -> np.ndarray:
    import torch
    if t.dtype == torch.uint32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    if t.dtype == torch.uint16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def u32(x):
    import torch
    return dev(np.asarray(x, dtype=np.uint32).view(np.int32)).view(torch.uint32)


def u16(x):
    import torch
    return dev(np.asarray(x, dtype=np.uint16).view(np.int16)).view(torch.uint16)


def logits_rows(cfg_V, rows, step, seed, sigma, boost, frac, dtype):
    """(exact float values for the oracle, device tensor for the kernel)."""
    import torch
    vals, raw = make_logits(cfg_V, rows, step, seed, sigma, boost, frac, dtype)
    if dtype == "bf16":
        t = dev(raw.view(np.int16)).view(torch.bfloat16)
    else:
        t = dev(raw)
    return vals.astype(np.float64), t


def oracle_bitmask(dfa, vm, state, forced=-1):
    from oracle.step import onehot_mask, token_mask
    if forced >= 0:
        return pack_bitmask(onehot_mask(vm.V, forced))
    return pack_bitmask(token_mask(dfa, vm, state))


def same_token(gpu_tok, res, tol=1e-5):
    """Sampled ids agree, except where the pages' tolerance admits either:
    top-two Gumbel scores closer than tol, or a top-p threshold within tol."""
    return gpu_tok == res.tok or res.gap < tol or res.margin < tol
