"""GB300-native grammar-constrained decoding: Python binding of libcg.so.

Every operation runs in the C/CUDA library (include/cg.h); this module only
marshals arguments: numpy arrays for host data, torch CUDA tensors (pointers
and the current stream) for device data.

    g = Grammar.compile(source, kind="json", bounds=Bounds())
    v = Vocab(list_of_token_bytes)
    ctx = Ctx([g], v)                        # binds torch's current CUDA stream
    ctx.fill_bitmask(states, bitmask, gid=None, forced=None)
    ctx.mask_and_sample(logits, bitmask, temp, top_p, seed, step, out_tok)
    ctx.accept(states, toks, out_states, out_flags)
"""

from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import _lib as L
from ._lib import (CG_DEAD, CG_FLAG_CAPPED, CG_FLAG_DONE, CG_FLAG_FORCED_NEXT,  # noqa: F401
                   CG_FLAG_NO_TOKEN, CG_FLAG_REJECTED, CG_NO_TOKEN, CG_STATE_ACCEPT,
                   CG_STATE_FORCED_ONLY, CG_STATE_SINK, CgError)


@dataclass(frozen=True)
class Bounds:
    ws_max: int = 4
    max_len_default: int = 256
    depth_max: int = 5
    max_items_default: int = 16
    max_tokens: int = 2048

    def c(self) -> L.cg_bounds:
        return L.cg_bounds(self.ws_max, self.max_len_default, self.depth_max, self.max_items_default,
                           self.max_tokens)


def _u32p(x):
    return C.byref(x)


class Grammar:
    def __init__(self, handle):
        self._h = C.c_void_p(handle)

    @classmethod
    def compile(cls, source: str | bytes, kind: str = "gbnf", bounds: Bounds = Bounds()) -> "Grammar":
        data = source.encode("utf-8") if isinstance(source, str) else bytes(source)
        out = C.c_void_p()
        err = C.create_string_buffer(512)
        k = {"gbnf": L.CG_GBNF, "json": L.CG_JSON_SCHEMA, "structtag": L.CG_STRUCTURAL_TAG}[kind]
        b = bounds.c()
        rc = L.lib().cg_compile(data, len(data), k, C.byref(b), C.byref(out), err, len(err))
        L.check("cg_compile", rc, err.value.decode("utf-8", "replace"))
        return cls(out.value)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_grammar_destroy(self._h)
            self._h = C.c_void_p()

    def info(self) -> dict:
        n, cols, start = C.c_uint32(), C.c_uint32(), C.c_uint32()
        L.check("cg_grammar_info", L.lib().cg_grammar_info(self._h, C.byref(n), C.byref(cols), C.byref(start)))
        return {"n_states": n.value, "n_cols": cols.value, "start": start.value}

    def export(self) -> tuple[np.ndarray, np.ndarray]:
        S = self.info()["n_states"]
        nxt = np.empty((S, 512), dtype=np.int32)
        flags = np.empty(S, dtype=np.uint8)
        L.check("cg_grammar_export", L.lib().cg_grammar_export(self._h, nxt.ctypes.data, flags.ctypes.data))
        return nxt, flags

    def try_input(self, data: bytes, injected: np.ndarray | None = None) -> tuple[int, int, bool]:
        ref, end, acc = C.c_size_t(), C.c_uint32(), C.c_int()
        inj = None
        if injected is not None:
            injected = np.ascontiguousarray(injected, dtype=np.uint8)
            inj = injected.ctypes.data
        L.check("cg_try_input", L.lib().cg_try_input(self._h, data, len(data), inj, C.byref(ref), C.byref(end),
                                                      C.byref(acc)))
        return ref.value, end.value, bool(acc.value)

    def live_states(self) -> np.ndarray:
        n = C.c_uint32()
        L.check("cg_live_states", L.lib().cg_live_states(self._h, None, 0, C.byref(n)))
        out = np.empty(n.value, dtype=np.uint32)
        L.check("cg_live_states", L.lib().cg_live_states(self._h, out.ctypes.data, n.value, C.byref(n)))
        return out


class Vocab:
    def __init__(self, tokens: list[bytes]):
        off = np.zeros(len(tokens) + 1, dtype=np.uint32)
        off[1:] = np.cumsum([len(t) for t in tokens])
        data = np.frombuffer(b"".join(tokens), dtype=np.uint8).copy()
        h = C.c_void_p()
        L.check("cg_vocab_create", L.lib().cg_vocab_create(data.ctypes.data, off.ctypes.data, len(tokens), C.byref(h)))
        self._h = h
        self.V = len(tokens)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_vocab_destroy(self._h)
            self._h = C.c_void_p()

    def tokenize_greedy(self, text: bytes) -> list[int]:
        out = np.empty(len(text) + 1, dtype=np.uint32)
        n = C.c_size_t()
        L.check("cg_tokenize_greedy", L.lib().cg_tokenize_greedy(self._h, text, len(text), out.ctypes.data,
                                                                  len(out), C.byref(n)))
        return out[:n.value].tolist()


def eval_arith(span: bytes, fmt: str) -> tuple[bytes, bool]:
    f = {"calc_tag": L.CG_RESULT_CALC_TAG, "json_answer": L.CG_RESULT_JSON_ANSWER}[fmt]
    buf = C.create_string_buffer(256)
    n, ok = C.c_size_t(), C.c_int()
    L.check("cg_eval_arith", L.lib().cg_eval_arith(span, len(span), f, buf, len(buf), C.byref(n), C.byref(ok)))
    return buf.raw[:n.value], bool(ok.value)


def mask_classes(grammars: list["Grammar"], max_len: int) -> tuple[np.ndarray, int]:
    """Joint mask classes of grammars used in one context: (class of every
    state, grammar after grammar; number of classes)."""
    arr = (C.c_void_p * len(grammars))(*[g._h.value for g in grammars])
    S, n = C.c_uint32(), C.c_uint32()
    L.check("cg_mask_classes", L.lib().cg_mask_classes(arr, len(grammars), max_len, None, 0, C.byref(S), C.byref(n)))
    out = np.zeros(S.value, dtype=np.uint32)
    L.check("cg_mask_classes", L.lib().cg_mask_classes(arr, len(grammars), max_len, out.ctypes.data, S.value,
                                                        C.byref(S), C.byref(n)))
    return out, n.value


def eval_strop(span: bytes) -> tuple[bytes, bool]:
    """A string operation's forced bytes (<result>V</result> or <result_error>code</result_error>)."""
    buf = C.create_string_buffer(256)
    n, ok = C.c_size_t(), C.c_int()
    L.check("cg_eval_strop", L.lib().cg_eval_strop(span, len(span), buf, len(buf), C.byref(n), C.byref(ok)))
    return buf.raw[:n.value], bool(ok.value)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


class Ctx:
    """Device context bound to one CUDA stream (torch's current stream by default)."""

    def __init__(self, grammars: list[Grammar], vocab: Vocab, stream=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        self.stream = stream
        arr = (C.c_void_p * len(grammars))(*[g._h.value for g in grammars])
        h = C.c_void_p()
        L.check("cg_ctx_create", L.lib().cg_ctx_create(arr, len(grammars), vocab._h, C.c_void_p(stream.cuda_stream),
                                                       C.byref(h)))
        self._h = h
        self.V = vocab.V
        self.W = (vocab.V + 31) // 32

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_ctx_destroy(self._h)
            self._h = C.c_void_p()

    def info(self) -> dict:
        nc, cb, V, W = C.c_uint32(), C.c_uint64(), C.c_uint32(), C.c_uint32()
        L.check("cg_ctx_info", L.lib().cg_ctx_info(self._h, C.byref(nc), C.byref(cb), C.byref(V), C.byref(W)))
        return {"n_classes": nc.value, "cache_bytes": cb.value, "V": V.value, "W": W.value}

    def status(self) -> int:
        code = C.c_uint32()
        rc = L.lib().cg_ctx_status(self._h, C.byref(code))
        if rc not in (L.CG_OK, L.CG_E_DEVICE):
            L.check("cg_ctx_status", rc)
        return code.value

    def prefill(self) -> None:
        L.check("cg_ctx_prefill", L.lib().cg_ctx_prefill(self._h))

    def cache_stats(self) -> dict:
        """Mask-cache counters (synchronises the stream): lookups and class masks
        computed by the segmented fused step's pre-pass, and the class masks in
        the cache now by any path ("ready", of info()["n_classes"])."""
        lk, cm, rd = C.c_uint64(), C.c_uint64(), C.c_uint32()
        L.check("cg_ctx_cache_stats", L.lib().cg_ctx_cache_stats(self._h, C.byref(lk), C.byref(cm), C.byref(rd)))
        return {"lookups": lk.value, "computed": cm.value, "ready": rd.value}

    def fill_bitmask(self, states, bitmask, gid=None, forced=None) -> None:
        B = states.shape[0]
        L.check("cg_fill_bitmask", L.lib().cg_fill_bitmask(self._h, _ptr(states), _ptr(gid), _ptr(forced), B,
                                                            _ptr(bitmask)))

    def mask_and_sample(self, logits, bitmask, temp: float, top_p: float, seed: int, step: int, out_tok,
                        probs=None, inplace: bool = False) -> None:
        import torch
        dtype = {torch.float32: L.CG_F32, torch.bfloat16: L.CG_BF16}[logits.dtype]
        B, V = logits.shape
        L.check("cg_mask_and_sample", L.lib().cg_mask_and_sample(
            self._h, _ptr(logits), dtype, B, V, _ptr(bitmask), float(temp), float(top_p), int(seed), int(step),
            _ptr(out_tok), _ptr(probs), L.CG_SAMPLE_INPLACE if inplace else 0))

    def mask_and_sample_noalloc(self, logits, bitmask, temp: float, top_p: float, seed: int, step: int, out_tok,
                                probs=None, inplace: bool = False) -> None:
        """mask_and_sample on the library's fixed scratch (no device allocation;
        B <= CG_NOALLOC_MAX_ROWS; overlapping calls on one device race)."""
        import torch
        dtype = {torch.float32: L.CG_F32, torch.bfloat16: L.CG_BF16}[logits.dtype]
        B, V = logits.shape
        L.check("cg_mask_and_sample_noalloc", L.lib().cg_mask_and_sample_noalloc(
            self._h, _ptr(logits), dtype, B, V, _ptr(bitmask), float(temp), float(top_p), int(seed), int(step),
            _ptr(out_tok), _ptr(probs), L.CG_SAMPLE_INPLACE if inplace else 0))

    def accept(self, states, toks, out_states, out_flags, gid=None, forced=None, counts=None,
               max_tokens: int = 2048) -> None:
        B = states.shape[0]
        L.check("cg_accept", L.lib().cg_accept(self._h, _ptr(states), _ptr(gid), _ptr(toks), _ptr(forced), B,
                                                _ptr(counts), max_tokens, _ptr(out_states), _ptr(out_flags)))


    def step(self, states, logits, temp: float, top_p: float, seed: int, step: int, out_tok, out_states, out_flags,
             gid=None, forced=None, counts=None, max_tokens: int = 2048, bitmask=None) -> None:
        """fill_bitmask + mask_and_sample + accept in one call (one segmented
        kernel for bf16 logits); bitmask, when given, receives the row masks."""
        import torch
        dtype = {torch.float32: L.CG_F32, torch.bfloat16: L.CG_BF16}[logits.dtype]
        B, V = logits.shape
        L.check("cg_step", L.lib().cg_step(
            self._h, _ptr(states), _ptr(gid), _ptr(forced), B, _ptr(logits), dtype, V, float(temp), float(top_p),
            int(seed), int(step), _ptr(counts), max_tokens, _ptr(bitmask), _ptr(out_tok), _ptr(out_states),
            _ptr(out_flags)))


    def accept_many(self, states, draft, draft_len, out_states, out_n, out_flags, gid=None, forced=None,
                    counts=None, max_tokens: int = 2048, path=None) -> None:
        """Speculative verification: the longest grammatical prefix of each row's
        draft ([B, K] ids, draft_len per row); forced [B, K] pins positions."""
        B, K = draft.shape
        L.check("cg_accept_many", L.lib().cg_accept_many(
            self._h, _ptr(states), _ptr(gid), _ptr(draft), _ptr(draft_len), _ptr(forced), B, K, _ptr(counts),
            max_tokens, _ptr(out_states), _ptr(out_n), _ptr(out_flags), _ptr(path)))

    def step_host(self, states, h_logits, temp: float, top_p: float, seed: int, step: int, h_out_tok, out_states,
                  out_flags, gid=None, forced=None, counts=None, max_tokens: int = 2048, out_tok=None) -> None:
        """cg_step with the logits in (page-locked) host memory and the ids
        copied back to host memory; asynchronous until sync()."""
        import torch
        dtype = {torch.float32: L.CG_F32, torch.bfloat16: L.CG_BF16}[h_logits.dtype]
        B, V = h_logits.shape
        L.check("cg_step_host", L.lib().cg_step_host(
            self._h, _ptr(states), _ptr(gid), _ptr(forced), B, _ptr(h_logits), dtype, V, float(temp), float(top_p),
            int(seed), int(step), _ptr(counts), max_tokens, _ptr(h_out_tok), _ptr(out_tok), _ptr(out_states),
            _ptr(out_flags)))

    def self_test_wait_timeout(self) -> None:
        """Make one bounded device wait run out (the status then reads CG_DEV_TIMEOUT)."""
        L.check("cg_self_test_wait_timeout", L.lib().cg_self_test_wait_timeout(self._h))

    def sync(self) -> None:
        L.check("cg_ctx_sync", L.lib().cg_ctx_sync(self._h))


class PdaGrammar:
    """A recursive GBNF grammar compiled to a pushdown automaton with a stack
    bound of ``depth`` frames (cg_pda_compile)."""

    def __init__(self, source: str | bytes, depth: int):
        data = source.encode("utf-8") if isinstance(source, str) else bytes(source)
        out = C.c_void_p()
        L.check("cg_pda_compile", L.lib().cg_pda_compile(data, len(data), int(depth), C.byref(out)))
        self._h = out

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_pda_grammar_destroy(self._h)
            self._h = C.c_void_p()

    def info(self) -> dict:
        n, r, cols, d = C.c_uint32(), C.c_uint32(), C.c_uint32(), C.c_uint32()
        L.check("cg_pda_grammar_info", L.lib().cg_pda_grammar_info(self._h, C.byref(n), C.byref(r), C.byref(cols),
                                                                    C.byref(d)))
        return {"n_states": n.value, "n_rules": r.value, "n_cols": cols.value, "depth": d.value}

    def try_input(self, data: bytes, injected: np.ndarray | None = None) -> tuple[int, bool, int]:
        """(bytes walked before the first refused one, complete, stack level)."""
        n, acc, lvl = C.c_size_t(), C.c_int(), C.c_uint32()
        inj = None
        if injected is not None:
            injected = np.ascontiguousarray(injected, dtype=np.uint8)
            inj = injected.ctypes.data
        L.check("cg_pda_try_input", L.lib().cg_pda_try_input(self._h, data, len(data), inj, C.byref(n),
                                                              C.byref(acc), C.byref(lvl)))
        return n.value, bool(acc.value), lvl.value


class Pda:
    """Pushdown rows on a context (cg_pda_create).  Row configurations are a
    u32 tensor [B, depth + 2]: state, stack level, return states."""

    def __init__(self, ctx: Ctx, vocab: Vocab, grammar: PdaGrammar):
        h = C.c_void_p()
        L.check("cg_pda_create", L.lib().cg_pda_create(ctx._h, vocab._h, grammar._h, C.byref(h)))
        self._h = h
        self._ctx = ctx  # destroyed before its context
        self.depth = grammar.info()["depth"]
        self.row_words = self.depth + 2

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_pda_destroy(self._h)
            self._h = C.c_void_p()

    def info(self) -> dict:
        k, m, cb, nc = C.c_uint32(), C.c_uint32(), C.c_uint64(), C.c_uint32()
        L.check("cg_pda_info", L.lib().cg_pda_info(self._h, C.byref(k), C.byref(m), C.byref(cb), C.byref(nc)))
        return {"n_keys": k.value, "n_masks": m.value, "cache_bytes": cb.value, "n_candidates": nc.value}

    def fill_bitmask(self, cfg, bitmask, forced=None) -> None:
        L.check("cg_pda_fill_bitmask", L.lib().cg_pda_fill_bitmask(self._h, _ptr(cfg), cfg.shape[0], _ptr(forced),
                                                                    _ptr(bitmask)))

    def accept(self, cfg, toks, out_flags, forced=None, counts=None, max_tokens: int = 0) -> None:
        L.check("cg_pda_accept", L.lib().cg_pda_accept(self._h, _ptr(cfg), cfg.shape[0], _ptr(toks), _ptr(forced),
                                                        _ptr(counts), int(max_tokens), _ptr(out_flags)))

    def step(self, cfg, logits, temp: float, top_p: float, seed: int, step: int, out_tok, out_flags, forced=None,
             counts=None, max_tokens: int = 0, bitmask=None) -> None:
        """mask, sample and accept in one call (one kernel on the bf16 top-p path)."""
        import torch
        dtype = {torch.float32: L.CG_F32, torch.bfloat16: L.CG_BF16}[logits.dtype]
        B, V = logits.shape
        L.check("cg_pda_step", L.lib().cg_pda_step(
            self._h, _ptr(cfg), B, _ptr(logits), dtype, V, float(temp), float(top_p), int(seed), int(step),
            _ptr(forced), _ptr(counts), int(max_tokens), _ptr(bitmask), _ptr(out_tok), _ptr(out_flags)))

    def accept_many(self, cfg, draft, draft_len, out_n, out_flags, forced=None, counts=None,
                    max_tokens: int = 0) -> None:
        """Speculative verification of drafts [B, K] against the rows' configurations."""
        B, K = draft.shape
        L.check("cg_pda_accept_many", L.lib().cg_pda_accept_many(
            self._h, _ptr(cfg), B, _ptr(draft), _ptr(draft_len), _ptr(forced), K, _ptr(counts), int(max_tokens),
            _ptr(out_n), _ptr(out_flags)))

    def accept_fill(self, cfg, toks, out_flags, bitmask, forced=None, counts=None, max_tokens: int = 0,
                    forced_next=None) -> None:
        """accept, then fill_bitmask of the next step, in one launch."""
        L.check("cg_pda_accept_fill", L.lib().cg_pda_accept_fill(
            self._h, _ptr(cfg), cfg.shape[0], _ptr(toks), _ptr(forced), _ptr(counts), int(max_tokens),
            _ptr(out_flags), _ptr(forced_next), _ptr(bitmask)))


class Driver:
    """Host driver of forced tokens (evaluator-aware grammars)."""

    def __init__(self, vocab: Vocab, B: int, gid: np.ndarray | None, rules: list[tuple[bytes, bytes, int]]):
        self._keep = []
        arr = (L.cg_span_rule * len(rules))()
        for i, (op, cl, fmt) in enumerate(rules):
            bo = C.create_string_buffer(op, len(op) or 1)
            bc = C.create_string_buffer(cl, len(cl) or 1)
            self._keep += [bo, bc]
            arr[i] = L.cg_span_rule(C.cast(bo, C.c_void_p), len(op), C.cast(bc, C.c_void_p), len(cl), fmt)
        g = None
        if gid is not None:
            self._gid = np.ascontiguousarray(gid, dtype=np.uint16)
            g = self._gid.ctypes.data
        h = C.c_void_p()
        L.check("cg_driver_create", L.lib().cg_driver_create(vocab._h, B, g, arr, len(rules), C.byref(h)))
        self._h = h
        self.B = B

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            L.lib().cg_driver_destroy(self._h)
            self._h = C.c_void_p()

    def update(self, toks: np.ndarray, flags: np.ndarray, forced_used: np.ndarray, forced_next: np.ndarray) -> int:
        n = C.c_uint32()
        L.check("cg_driver_update", L.lib().cg_driver_update(self._h, toks.ctypes.data, flags.ctypes.data,
                                                              forced_used.ctypes.data, forced_next.ctypes.data,
                                                              C.byref(n)))
        return n.value
