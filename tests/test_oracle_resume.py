"""The oracle's state is all in the caller's arrays: 10 steps equal 5 steps,
a save of master/m/v to a file, a reload and 5 more steps, bit for bit."""
import numpy as np

from fsdp_sharded_mixed_flatten_gb300 import synthetic

HP = dict(synthetic.ADAMW_DEFAULTS)


def _grads(P, n, t):
    return synthetic.bf16_bits(synthetic.make_grads(P, n, 1e-2, ("oracle-resume", t)))


def test_oracle_resume_is_bit_exact(oracle, tmp_path):
    P, n = 1003, 4
    S = -(-P // n)
    m0 = synthetic.make_master_flat(P, n, 0.02, ("oracle-resume",)).numpy().reshape(n, S)
    a = [m0.copy(), np.zeros_like(m0), np.zeros_like(m0)]
    for t in range(1, 11):
        out_a = oracle.zero_step(_grads(P, n, t), *a, step=t, **HP)
    b = [m0.copy(), np.zeros_like(m0), np.zeros_like(m0)]
    for t in range(1, 6):
        oracle.zero_step(_grads(P, n, t), *b, step=t, **HP)
    np.savez(tmp_path / "state.npz", master=b[0], m=b[1], v=b[2])
    z = np.load(tmp_path / "state.npz")
    c = [z["master"].copy(), z["m"].copy(), z["v"].copy()]
    for t in range(6, 11):
        out_c = oracle.zero_step(_grads(P, n, t), *c, step=t, **HP)
    for x, y in zip(a, c):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert np.array_equal(out_a, out_c)
