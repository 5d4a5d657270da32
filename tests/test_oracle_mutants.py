"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of the oracle's C source with one plausible slip
(compiled on the CPU into a temporary directory); the pin tests (PIN_FILES)
are rerun against it and at least one must fail.  The
allocator model gets the same treatment through small subclasses.
"""
import os
import subprocess
import sys

import pytest

import oracle
from oracle import alloc_model

HERE = os.path.dirname(os.path.abspath(__file__))

C_MUTANTS = {
    "scale_dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
    "offset_uses_block_index": ("(size_t)(t % block_size)) * head_dim;", "(size_t)(t / block_size)) * head_dim;"),
    "logical_used_as_physical": ("int32_t phys = table[t / block_size];", "int32_t phys = t / block_size;"),
    "kv_head_reversed": ("* num_kv_heads + g) * block_size", "* num_kv_heads + (num_kv_heads - 1 - g)) * block_size"),
    "query_row_from_kv_head": ("size_t qrow = ((size_t)b * num_q_heads + h) * head_dim;\n                double m",
                               "size_t qrow = ((size_t)b * num_q_heads + g) * head_dim;\n                double m"),
    "softmax_not_normalised": ("double w = s[t] / denom;", "double w = s[t];"),
    "reduce_weight_inverted": ("double w = exp(m[p] - M);", "double w = exp(M - m[p]);"),
    "reduce_drops_l": ("L += w * l[p];", "L += w;"),
    "partition_max_unscaled": ("if (scale * dot > m) m = scale * dot;", "if (dot > m) m = dot;"),
    "prefill_position_ignores_context": ("const int32_t p = len - n + i;", "const int32_t p = i;"),
    "prefill_position_one_early": ("const int32_t p = len - n + i;", "const int32_t p = len - n + i - 1;"),
    "prefill_rows_reversed": ("const size_t row = (size_t)cu_q_lens[b] + (size_t)i;",
                              "const size_t row = (size_t)cu_q_lens[b + 1] - 1 - (size_t)i;"),
    "prefill_not_causal": ("for (int32_t t = 0; t <= p; ++t) {\n                        double dot",
                           "for (int32_t t = 0; t < len; ++t) {\n                        double dot"),
    "e4m3_ties_to_odd": ("(dc == db && (c & 1) == 0 && (best & 1) == 1)", "(dc == db && (c & 1) == 1 && (best & 1) == 0)"),
    "e4m3_subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_saturates_at_416": ("for (int c = 1; c <= 0x7E; ++c) {", "for (int c = 1; c <= 0x7D; ++c) {"),
    "append_slot_before_head": ("size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * head_dim + e;",
                                "size_t dst = (((size_t)blk * block_size + (size_t)off) * num_kv_heads + h) * head_dim + e;"),
    "append_k_only": ("memcpy((char*)v_pool + dst * elem_bytes, (const char*)v_new + src * elem_bytes, elem_bytes);", ""),
    "append_skips_slot_zero": ("if (s < 0) continue;\n        int64_t blk = s / block_size, off = s % block_size;",
                               "if (s <= 0) continue;\n        int64_t blk = s / block_size, off = s % block_size;"),
    "append_offset_from_block": ("int64_t blk = s / block_size, off = s % block_size;",
                                 "int64_t blk = s / block_size, off = blk % block_size;"),
    "copy_k_only": ("memcpy((char*)v_pool + ((size_t)dst * block_elems + e) * elem_bytes,\n"
                    "                   (const char*)v_pool + ((size_t)src * block_elems + e) * elem_bytes, elem_bytes);", ""),
    "copy_one_head": ("for (size_t e = 0; e < block_elems; ++e) {", "for (size_t e = 0; e < block_elems / num_kv_heads; ++e) {"),
    "copy_direction_reversed": ("int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];",
                                "int32_t dst = pairs[2 * p], src = pairs[2 * p + 1];"),
    "fp8_v_scale_dropped": ("V[(size_t)t * head_dim + i] = load_elem(dtype, v_pool, row + i) * v_scale;",
                            "V[(size_t)t * head_dim + i] = load_elem(dtype, v_pool, row + i);"),
}
PIN_FILES = ["test_oracle_pins.py", "test_oracle_prefill_pins.py", "test_oracle_fp8_pins.py",
             "test_oracle_cache_ops_pins.py"]


@pytest.fixture(scope="module")
def src():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_mutant_is_caught(name, src, tmp_path):
    old, new = C_MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "mut.c"
    c.write_text(mutated)
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"])
    # run the pin tests in a child process whose oracle loads the mutant
    code = (
        "import sys, pytest, oracle;"
        f"oracle._lib = oracle._open({str(so)!r});"
        f"sys.exit(pytest.main(['-q', '-x', '-p', 'no:cacheprovider', *{[os.path.join(HERE, f) for f in PIN_FILES]!r}]))"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=os.path.dirname(HERE), capture_output=True, text=True,
                       env={**os.environ, "PYTHONPATH": os.pathsep.join([os.path.dirname(HERE), HERE])})
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"


class _CowOnAnyRef(alloc_model.RefAllocator):
    def _append_one(self, sid, slots, pairs):  # copies even a private tail
        table = self.tables[sid]
        n = self.lens[sid]
        if n % self.block_size and self.ref[table[-1]] >= 1 and len(table) > 1:
            fresh = self._take()
            pairs.append((table[-1], fresh))
            self.ref[table[-1]] -= 1
            table[-1] = fresh
        elif n % self.block_size == 0:
            table.append(self._take())
        slots.append(table[n // self.block_size] * self.block_size + n % self.block_size)
        self.lens[sid] = n + 1


class _LifoFree(alloc_model.RefAllocator):
    def free_seq(self, sid):
        for b in self.tables[sid]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.appendleft(b)
        del self.tables[sid]
        del self.lens[sid]


class _ForkNoRef(alloc_model.RefAllocator):
    def fork(self, parent, child):
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]


@pytest.mark.parametrize("cls", [_CowOnAnyRef, _LifoFree, _ForkNoRef])
def test_alloc_model_mutant_is_caught(cls):
    from test_alloc_model import run_trace

    with pytest.raises(AssertionError):
        run_trace(lambda nb, bs, order: cls(nb, bs, free_order=order))
