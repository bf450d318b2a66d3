"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function ``include/tp.h`` declares, and its host-only validation and
shard tables agree bit-exactly with the oracle's independent computation.
No compute call is made (there is no GPU here)."""
import ctypes as C
import os
import re

import pytest

import oracle
import megatron_tensor_transformer_colwise_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tp.h")).read()
    return sorted(set(re.findall(r"^TP_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("tp_plan_create", "tp_mlp_forward", "tp_attn_forward", "tp_reduce_partials",
                 "tp_layer_forward"):
        assert must in names
    assert tuple(names) == tp.EXPORTED   # binding covers exactly the header


def declared_arg_counts():
    """Number of parameters of every TP_API declaration in tp.h."""
    src = open(os.path.join(ROOT, "include", "tp.h")).read()
    out = {}
    for m in re.finditer(r"^TP_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(([^)]*)\)", src, flags=re.M):
        params = " ".join(m.group(2).split())
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_the_header():
    counts = declared_arg_counts()
    assert set(counts) == set(tp.EXPORTED)
    for name, args in tp._SIGS.items():
        assert len(args) == counts[name], f"{name}: binding {len(args)} args, header {counts[name]}"


def test_library_exports_every_declared_symbol():
    L = tp.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
        assert C.cast(getattr(L, name), C.c_void_p).value


def test_library_is_built_for_sm_103a_only():
    from megatron_tensor_transformer_colwise_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(_build.LIB)


def cfg(**kw):
    base = dict(tokens=64, hidden=64, ffn=256, n_heads=8, n_kv_heads=8, head_dim=64, tp_degree=4,
                act="gelu", batch=1, seq=64)
    base.update(kw)
    return tp.make_config(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(), tp.TP_OK),
    (dict(tp_degree=3), tp.TP_ERR_NOT_DIVISIBLE),                  # t does not divide f or a
    (dict(ffn=250), tp.TP_ERR_NOT_DIVISIBLE),                      # t does not divide f
    (dict(ffn=96), tp.TP_OK),                                      # f/t = 24, a multiple of 8
    (dict(ffn=72), tp.TP_ERR_INVALID_ARG),                         # f/t = 18 breaks 16-byte rows
    (dict(n_heads=12, n_kv_heads=4), tp.TP_OK),                    # t | a, k | a, t | k
    (dict(n_heads=12, n_kv_heads=12, tp_degree=8, ffn=256), tp.TP_ERR_NOT_DIVISIBLE),  # t does not divide a
    (dict(n_heads=8, n_kv_heads=3), tp.TP_ERR_NOT_DIVISIBLE),      # k does not divide a
    (dict(n_heads=16, n_kv_heads=2, tp_degree=4, ffn=256), tp.TP_OK),  # k < t, replicas
    (dict(n_heads=24, n_kv_heads=6, tp_degree=4, ffn=256), tp.TP_ERR_NOT_DIVISIBLE),  # k>=t, t∤k
    (dict(head_dim=96), tp.TP_ERR_UNSUPPORTED),
    (dict(hidden=60), tp.TP_ERR_INVALID_ARG),
    (dict(tokens=0, seq=0), tp.TP_ERR_INVALID_ARG),
    (dict(tokens=64, batch=2, seq=16), tp.TP_ERR_INVALID_ARG),      # tokens != batch * seq
    (dict(act=7), tp.TP_ERR_INVALID_ARG),
    (dict(reduce_mode=5), tp.TP_ERR_INVALID_ARG),
    (dict(partial_dtype=tp.TP_BF16), tp.TP_ERR_UNSUPPORTED),        # bf16 partials need PARTIALS mode
    (dict(partial_dtype=tp.TP_BF16, reduce_mode=tp.TP_REDUCE_PARTIALS), tp.TP_OK),
    (dict(tp_degree=0), tp.TP_ERR_INVALID_ARG),
    (dict(tp_degree=65), tp.TP_ERR_INVALID_ARG),
])
def test_config_check_codes(kw, want):
    c = cfg(**kw)
    got = tp.tp_config_check(c)
    assert got == want, tp.tp_last_error()
    if want != tp.TP_OK:
        assert tp.tp_last_error() and tp.tp_last_error() != "no error"


def test_config_check_agrees_with_oracle_on_divisibility():
    for t in (1, 2, 3, 4, 6, 8):
        for a, k in ((8, 8), (8, 2), (32, 8), (12, 3), (16, 1), (24, 6)):
            for f in (96, 240, 384):
                c = cfg(tp_degree=t, n_heads=a, n_kv_heads=k, ffn=f, head_dim=64)
                ours = tp.tp_config_check(c)
                ref = oracle.plan_check(64, f, a, k, 64, t)
                if ref == oracle.ERR_NOT_DIVISIBLE:
                    assert ours == tp.TP_ERR_NOT_DIVISIBLE, (t, a, k, f)
                elif ref == oracle.OK:
                    # the library adds its own alignment rule: (f/t) % 8 == 0
                    assert ours == (tp.TP_OK if (f // t) % 8 == 0 else tp.TP_ERR_INVALID_ARG), (t, a, k, f)


@pytest.mark.parametrize("a,k,t", [(32, 8, 8), (8, 2, 4), (16, 1, 8), (8, 8, 2), (24, 6, 3)])
def test_shard_tables_bit_exact_vs_oracle(a, k, t):
    f = 64 * t
    c = cfg(tp_degree=t, n_heads=a, n_kv_heads=k, ffn=f, head_dim=128)
    d = 128
    assert tp.tp_config_check(c) == tp.TP_OK, tp.tp_last_error()
    ffn = tp.tp_config_shard_table(c, tp.TP_TABLE_FFN_SHARDS)
    assert ffn == [v for i in range(t) for v in (i * (f // t), f // t)]
    qs = tp.tp_config_shard_table(c, tp.TP_TABLE_Q_HEAD_SHARD)
    assert qs == [oracle.q_head_shard(a, t, j) for j in range(a)]
    qk = tp.tp_config_shard_table(c, tp.TP_TABLE_Q_HEAD_KV)
    assert qk == [oracle.q_head_kv(a, k, j) for j in range(a)]
    skv = tp.tp_config_shard_table(c, tp.TP_TABLE_SHARD_KV)
    assert skv == [v for i in range(t) for v in (oracle.shard_kv_first(k, t, i),
                                                  oracle.shard_kv_count(k, t))]
    cols = tp.tp_config_shard_table(c, tp.TP_TABLE_QKV_COLUMNS)
    ap, kvn = a // t, oracle.shard_kv_count(k, t)
    w = (ap + 2 * kvn) * d
    assert cols == [v for i in range(t) for v in (i * w, i * w + ap * d, i * w + ap * d + kvn * d)]


def test_shard_table_rejects_unknown_and_small_capacity():
    c = cfg()
    n = C.c_int64(0)
    buf = (C.c_int32 * 2)()
    rc = tp.lib().tp_config_shard_table(C.byref(c), tp.TP_TABLE_Q_HEAD_SHARD, buf, 2, C.byref(n))
    assert rc == tp.TP_ERR_INVALID_ARG and n.value == 8
    rc = tp.lib().tp_config_shard_table(C.byref(c), 99, buf, 2, C.byref(n))
    assert rc == tp.TP_ERR_INVALID_ARG


def test_entry_points_reject_null_plan_without_touching_a_gpu():
    L = tp.lib()
    assert L.tp_mlp_forward(*([None] * 10), 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_attn_forward(*([None] * 10), 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_layer_forward(None, None, None, None, None, 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_reduce_partials(None, 0, 4, 64, 8, None, None, None, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_plan_create(None, None) == tp.TP_ERR_INVALID_ARG


@pytest.mark.parametrize("blocks,t", [([4, 4], 2), ([256, 256], 4), ([192, 192, 192, 576, 576], 3),
                                      ([64], 1), ([128, 64, 64], 8)])
def test_packed_shard_table_bit_exact_vs_oracle(blocks, t):
    if any(b % t for b in blocks):
        pytest.skip("not divisible")
    table = tp.tp_packed_shard_table(blocks, t)
    nb = len(blocks)
    for i in range(t):
        rows = []
        for b in range(nb):
            first, count = table[(i * nb + b) * 2], table[(i * nb + b) * 2 + 1]
            rows.extend(range(first, first + count))
        assert rows == oracle.packed_shard_rows(blocks, t, i).tolist()


def test_packed_shard_table_rejects_blocks_not_divisible_individually():
    with pytest.raises(tp.TPError) as e:
        tp.tp_packed_shard_table([6, 2], 4)
    assert e.value.code == tp.TP_ERR_NOT_DIVISIBLE
    assert "each block" in tp.tp_last_error()
    with pytest.raises(tp.TPError) as e:
        tp.tp_packed_shard_table([4] * 9, 2)
    assert e.value.code == tp.TP_ERR_INVALID_ARG


def test_sequence_parallel_config_rules():
    ok = cfg(tokens=64, batch=2, seq=32, tp_degree=4, reduce_mode=tp.TP_REDUCE_PARTIALS,
             sequence_parallel=1)
    assert tp.tp_config_check(ok) == tp.TP_OK, tp.tp_last_error()
    bad_seq = cfg(tokens=60, batch=2, seq=30, tp_degree=4, reduce_mode=tp.TP_REDUCE_PARTIALS,
                  sequence_parallel=1, ffn=256)
    assert tp.tp_config_check(bad_seq) == tp.TP_ERR_NOT_DIVISIBLE
    # FUSED mode: the reduce-scatter happens in the rowwise GEMM's accumulator.
    fused = cfg(tokens=64, batch=2, seq=32, tp_degree=4, sequence_parallel=1)
    assert tp.tp_config_check(fused) == tp.TP_OK, tp.tp_last_error()
    bad_tokens = cfg(tokens=64, batch=2, seq=16, tp_degree=4, sequence_parallel=1)
    assert tp.tp_config_check(bad_tokens) == tp.TP_ERR_INVALID_ARG
