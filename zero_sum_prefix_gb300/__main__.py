from zero_sum_prefix_gb300.build import build

print(build(verbose=True))
