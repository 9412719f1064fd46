set -e
cd _work/tl
for pf in 0 1 2; do nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I ../../include -DPF=$pf -o tl_pf$pf main_tl.cu 2>/dev/null; done
for pf in 1 0 2; do echo "=== PF=$pf"; ./tl_pf$pf 1 | grep -v "^ *$"; done
